"""Host-side metadata checks (msgl_check_*_meta) on CPU: valid steps pass, planted mistakes are named.

The checks read host copies, so these tests run without a GPU.  The valid
metadata comes from the seeded workloads; each mistake is planted in a copy.
"""
import pytest
import torch

from paged_kv_attention_24_gb300 import ops
from paged_kv_attention_24_gb300 import workloads as W

INVALID, OUT_OF_RANGE = 1, 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    from paged_kv_attention_24_gb300 import build
    build.build()
    return ops.load()


@pytest.fixture(scope="module")
def c1():
    return W.config(1, device="cpu")


@pytest.fixture(scope="module")
def c2():
    return W.config(2, device="cpu")


def expect(status, fragment, fn, *args):
    with pytest.raises(ops.MsglError) as e:
        fn(*args)
    assert e.value.status == status, str(e.value)
    assert fragment in str(e.value), str(e.value)


def ext_args(w, **over):
    e = w.extend
    args = dict(num_slots=w.num_slots, page_size=w.page_size, page_table=e.page_table.clone(),
                prefix_lens=e.prefix_lens.clone(), ext_lens=e.ext_lens.clone(), cu_ext=e.cu_ext.clone(),
                positions=e.positions.clone(), max_ext_len=e.max_ext_len, max_seq_len=e.max_seq_len)
    args.update(over)
    return args


def test_workload_metadata_passes(c1, c2):
    d = c1.decode
    ops.check_decode_meta(c1.num_slots, c1.page_size, d.page_table, d.seq_lens, d.max_seq_len)
    ops.check_extend_meta(**ext_args(c2))
    ops.check_extend_meta(**ext_args(c2, positions=None))
    for w in (c1, c2):
        _, _, loc = w.new_tokens()
        ops.check_store_meta(loc, w.num_slots)


def test_store_duplicate_and_range(c2):
    _, _, loc = c2.new_tokens()
    dup = loc.clone()
    dup[7] = dup[3]
    expect(INVALID, "out_loc[7]", ops.check_store_meta, dup, c2.num_slots)
    far = loc.clone()
    far[5] = c2.num_slots
    expect(OUT_OF_RANGE, "out_loc[5]", ops.check_store_meta, far, c2.num_slots)
    neg = loc.clone()
    neg[0] = -1
    expect(OUT_OF_RANGE, "out_loc[0]", ops.check_store_meta, neg, c2.num_slots)


def test_extend_position_off_by_one(c2):
    a = ext_args(c2)
    row = int(a["cu_ext"][3]) + 5
    a["positions"][row] += 1
    expect(INVALID, "request 3 row 5", ops.check_extend_meta, *a.values())


def test_extend_lengths(c2):
    a = ext_args(c2)
    a["cu_ext"][2] += 1
    expect(INVALID, "cu_ext", ops.check_extend_meta, *a.values())
    a = ext_args(c2, max_ext_len=int(c2.extend.ext_lens.max()) - 1)
    expect(INVALID, "max_ext_len", ops.check_extend_meta, *a.values())
    a = ext_args(c2, max_seq_len=int((c2.extend.prefix_lens + c2.extend.ext_lens).max()) - 1)
    expect(INVALID, "max_seq_len", ops.check_extend_meta, *a.values())
    a = ext_args(c2)
    a["prefix_lens"][1] = -4
    expect(INVALID, "request 1", ops.check_extend_meta, *a.values())


def test_extend_pages(c2):
    a = ext_args(c2)
    a["page_table"][4, 10] = c2.num_slots // c2.page_size
    expect(OUT_OF_RANGE, "request 4: page_ids[10]", ops.check_extend_meta, *a.values())
    # an entry past the request's last key is never read, so anything may sit there
    a = ext_args(c2)
    n = int(c2.extend.prefix_lens[0] + c2.extend.ext_lens[0])
    if n < a["page_table"].shape[1]:
        a["page_table"][0, n:] = -7
        ops.check_extend_meta(*a.values())
    # a table too narrow for the longest request
    a = ext_args(c2)
    need = int((c2.extend.prefix_lens + c2.extend.ext_lens).max())
    a["page_table"] = a["page_table"][:, :need - 1].contiguous()
    expect(OUT_OF_RANGE, "table width", ops.check_extend_meta, *a.values())


def test_decode_lengths_and_pages(c1):
    d = c1.decode
    seq = d.seq_lens.clone()
    seq[2] = 0
    expect(INVALID, "request 2: seq_len 0", ops.check_decode_meta, c1.num_slots, c1.page_size, d.page_table,
           seq, d.max_seq_len)
    expect(INVALID, "max_seq_len", ops.check_decode_meta, c1.num_slots, c1.page_size, d.page_table, d.seq_lens,
           int(d.seq_lens.max()) - 1)
    pt = d.page_table.clone()
    pt[1, int(d.seq_lens[1]) - 1] = -1
    expect(OUT_OF_RANGE, "request 1", ops.check_decode_meta, c1.num_slots, c1.page_size, pt, d.seq_lens,
           d.max_seq_len)


def test_bad_scalars():
    z = torch.zeros(2, dtype=torch.int32)
    expect(INVALID, "page_size", ops.check_decode_meta, 64, 3, z.reshape(1, 2), torch.ones(1, dtype=torch.int32), 4)
    expect(INVALID, "multiple of page_size", ops.check_decode_meta, 65, 4, z.reshape(1, 2),
           torch.ones(1, dtype=torch.int32), 4)
