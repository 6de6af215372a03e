"""The C-ABI library builds, loads and exports every declared entry point (CPU only).

Nothing here launches a kernel: the calls below fail host-side validation
(or are pure size queries) before any CUDA call is made.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_24_gb300 import build, ops
    build.build()
    return ops.load()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MSGL_API\s+[\w\s\*]+?\b(msgl_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("msgl_store_kv", "msgl_attn_extend", "msgl_attn_decode", "msgl_decode_workspace_size",
              "msgl_extend_workspace_size", "msgl_read_status", "msgl_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_signatures_cover_the_header():
    from paged_kv_attention_24_gb300 import ops, radix
    assert set(declared_functions()) <= set(ops.SIGNATURES) | set(radix.SIGNATURES)


def test_version_and_strings(lib):
    assert lib.msgl_abi_version() == 1
    assert lib.msgl_status_string(0) == b"ok"
    assert lib.msgl_status_string(6).startswith(b"workspace")
    assert lib.msgl_status_string(99) == b"unknown status"


def test_host_validation_needs_no_gpu(lib):
    from paged_kv_attention_24_gb300 import ops
    # NULL pool
    rc = lib.msgl_attn_decode(None, None, None, 16, None, 1, 10, 0.1, None, None, None, 0, None, None)
    assert rc == 1 and b"pool" in lib.msgl_last_error()
    # head_dim 64 is unsupported
    pool = ops._Pool(16, 16, 64, 1, 8, 64)
    rc = lib.msgl_store_kv(ctypes.byref(pool), 16, 16, 16, 1, None, None)
    assert rc == 2
    # page size not a power of two
    pool = ops._Pool(16, 16, 96, 3, 8, 128)
    rc = lib.msgl_store_kv(ctypes.byref(pool), 16, 16, 16, 1, None, None)
    assert rc == 2
    # misaligned pool
    pool = ops._Pool(18, 16, 64, 1, 8, 128)
    rc = lib.msgl_store_kv(ctypes.byref(pool), 16, 16, 16, 1, None, None)
    assert rc == 1
    # q heads not a multiple of kv heads; bad scale
    pool = ops._Pool(16, 16, 64, 1, 8, 128)
    pages = ops._Pages(16, 4, 4)
    rc = lib.msgl_attn_decode(ctypes.byref(pool), ctypes.byref(pages), 16, 12, 16, 1, 10, 0.1, 16, 16,
                              None, 0, None, None)
    assert rc == 1
    rc = lib.msgl_attn_decode(ctypes.byref(pool), ctypes.byref(pages), 16, 16, 16, 1, 10, -1.0, 16, 16,
                              None, 0, None, None)
    assert rc == 1
    # more than 64 q heads per kv head is unsupported (8 kv heads here)
    rc = lib.msgl_attn_decode(ctypes.byref(pool), ctypes.byref(pages), 16, 8 * 72, 16, 1, 10, 0.1, 16, 16,
                              None, 0, None, None)
    assert rc == 2
    # a split decode without workspace
    rc = lib.msgl_attn_decode(ctypes.byref(pool), ctypes.byref(pages), 16, 16, 16, 1, 100000, 0.1, 16,
                              16, None, 0, None, None)
    assert rc == 6
    # read_status on NULL
    assert lib.msgl_read_status(None, None, None) == 1
    # empty calls are no-ops
    assert lib.msgl_store_kv(ctypes.byref(pool), None, None, None, 0, None, None) == 0


def test_workspace_size_queries(lib):
    small = lib.msgl_decode_workspace_size(4, 16, 8, 128, 200)
    big = lib.msgl_decode_workspace_size(256, 16, 8, 128, 2048)
    assert big >= small >= 0
    assert lib.msgl_decode_workspace_size(4, 16, 8, 64, 200) == 0   # unsupported head_dim
    assert lib.msgl_decode_workspace_size(0, 16, 8, 128, 200) == 0
    assert big % 256 == 0


def test_noalloc_scratch_size_agrees_with_binding(lib):
    """The Python copy of the built-in scratch size equals the header's macro and the size
    the library itself reports when it refuses an over-size batch (a host-side check made
    before any CUDA call)."""
    from paged_kv_attention_24_gb300 import ops
    text = open(os.path.join(ROOT, "include", "msgl_attn.h")).read()
    m = re.search(r"#define MSGL_DECODE_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == ops.NOALLOC_SCRATCH_BYTES
    pool = ops._Pool(16, 16, 4096, 64, 8, 128)
    pages = ops._Pages(16, 64, 64)
    rc = lib.msgl_attn_decode_noalloc(ctypes.byref(pool), ctypes.byref(pages), 16, 64, 16, 600, 4096, 0.1,
                                      16, 16, None, None)
    assert rc == 6
    need = lib.msgl_decode_workspace_size(600, 64, 8, 128, 4096)
    msg = lib.msgl_last_error().decode()
    assert f"needs {need} scratch bytes" in msg and f"holds {ops.NOALLOC_SCRATCH_BYTES}" in msg, msg


def test_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structures have the C structs' sizes and field offsets
    (a C program built against include/msgl_attn.h prints them)."""
    import subprocess
    from paged_kv_attention_24_gb300 import ops
    src = tmp_path / "layout.c"
    structs = {"msgl_kv_pool": (ops._Pool, ["k_pool", "v_pool", "num_slots", "page_size", "num_kv_heads",
                                            "head_dim"]),
               "msgl_page_table": (ops._Pages, ["page_ids", "stride", "width"]),
               "msgl_extend_batch": (ops._ExtendBatch, ["pages", "q", "prefix_lens", "ext_lens", "cu_ext",
                                                        "positions", "num_reqs", "total_tokens", "max_ext_len",
                                                        "max_seq_len", "o", "lse"]),
               "msgl_decode_batch": (ops._DecodeBatch, ["pages", "q", "seq_lens", "num_reqs", "max_seq_len",
                                                        "o", "lse"])}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "msgl_attn.h"', "int main(void) {"]
    for name, (_, fields) in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for f in fields:
            lines.append(f'printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["return 0;", "}"]
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        name, field, value = line.split()
        got[(name, field)] = int(value)
    for name, (cls, fields) in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for f in fields:
            assert got[(name, f)] == getattr(cls, f).offset, (name, f)
