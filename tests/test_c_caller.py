"""The C ABI from a C program: no Python and no PyTorch on the call path.

A small C program, built against include/msgl_attn.h and linked with
libmsgl_attn.so, allocates device buffers with cudaMalloc, copies seeded inputs
in, calls msgl_store_kv, msgl_attn_extend and msgl_attn_decode with plain
pointers on a stream it created, reads the status word, and writes the outputs
to a file.  Python only prepares the input file (from the seeded generators)
and compares the outputs with the fp64 oracle.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_24_gb300 import build as cuda_build
from paged_kv_attention_24_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <stdint.h>
#include <cuda_runtime.h>
#include "msgl_attn.h"

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 2; } } while (0)
#define MK(x) do { msgl_status s_ = (x); if (s_ != MSGL_OK) { \
    fprintf(stderr, "%s: %s (%s)\n", #x, msgl_status_string(s_), msgl_last_error()); return 3; } } while (0)

static void *read_blob(FILE *f, size_t n) {
    void *p = malloc(n ? n : 1);
    if (n && fread(p, 1, n, f) != n) { fprintf(stderr, "short read\n"); exit(4); }
    return p;
}

static void *to_device(FILE *f, size_t n) {
    void *h = read_blob(f, n), *d = NULL;
    if (cudaMalloc(&d, n ? n : 16) != cudaSuccess) exit(5);
    if (n) cudaMemcpy(d, h, n, cudaMemcpyHostToDevice);
    free(h);
    return d;
}

int main(int argc, char **argv) {
    if (argc != 3) return 1;
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 1;
    int32_t hdr[10];
    if (fread(hdr, sizeof hdr, 1, f) != 1) return 4;
    const int64_t slots = hdr[0];
    const int32_t ps = hdr[1], hkv = hdr[2], hq = hdr[3], n_new = hdr[4];
    const int32_t eb = hdr[5], et = hdr[6], db = hdr[7], ew = hdr[8], dw = hdr[9];
    float scale;
    if (fread(&scale, sizeof scale, 1, f) != 1) return 4;
    int32_t lim[4];   /* max_ext_len, max_seq_len (extend), max_seq_len (decode), pad */
    if (fread(lim, sizeof lim, 1, f) != 1) return 4;
    const size_t row = (size_t)hkv * 128 * 2;
    void *kp = to_device(f, slots * row), *vp = to_device(f, slots * row);
    void *kn = to_device(f, n_new * row), *vn = to_device(f, n_new * row);
    void *loc = to_device(f, n_new * 4);
    void *eq = to_device(f, (size_t)et * hq * 256), *ept = to_device(f, (size_t)eb * ew * 4);
    void *pre = to_device(f, eb * 4), *ext = to_device(f, eb * 4), *cu = to_device(f, (eb + 1) * 4);
    void *pos = to_device(f, (size_t)et * 4);
    void *dq = to_device(f, (size_t)db * hq * 256), *dpt = to_device(f, (size_t)db * dw * 4);
    void *seq = to_device(f, db * 4);
    fclose(f);
    void *eo, *e_lse, *dout, *dlse, *status;
    CK(cudaMalloc(&eo, (size_t)et * hq * 256));
    CK(cudaMalloc(&e_lse, (size_t)et * hq * 4));
    CK(cudaMalloc(&dout, (size_t)db * hq * 256));
    CK(cudaMalloc(&dlse, (size_t)db * hq * 4));
    CK(cudaMalloc(&status, 4));
    CK(cudaMemset(status, 0, 4));
    cudaStream_t st;
    CK(cudaStreamCreate(&st));

    msgl_kv_pool pool = {kp, vp, slots, ps, hkv, 128};
    MK(msgl_store_kv(&pool, kn, vn, (const int32_t *)loc, n_new, (uint32_t *)status, st));
    msgl_page_table ept_t = {(const int32_t *)ept, ew, ew};
    const size_t ews = msgl_extend_workspace_size(eb, et, hq, hkv, 128, lim[1]);
    void *ewsp = NULL;
    if (ews) CK(cudaMalloc(&ewsp, ews));
    MK(msgl_attn_extend(&pool, &ept_t, eq, hq, (const int32_t *)pre, (const int32_t *)ext, (const int32_t *)cu,
                        (const int32_t *)pos, eb, et, lim[0], lim[1], scale, eo, (float *)e_lse, ewsp, ews,
                        (uint32_t *)status, st));
    msgl_page_table dpt_t = {(const int32_t *)dpt, dw, dw};
    const size_t dws = msgl_decode_workspace_size(db, hq, hkv, 128, lim[2]);
    void *dwsp = NULL;
    CK(cudaMalloc(&dwsp, dws));
    MK(msgl_attn_decode(&pool, &dpt_t, dq, hq, (const int32_t *)seq, db, lim[2], scale, dout, (float *)dlse,
                        dwsp, dws, (uint32_t *)status, st));
    uint32_t flags = 0;
    MK(msgl_read_status((const uint32_t *)status, &flags, st));

    size_t n_eo = (size_t)et * hq * 256, n_el = (size_t)et * hq * 4;
    size_t n_do = (size_t)db * hq * 256, n_dl = (size_t)db * hq * 4;
    char *buf = (char *)malloc(n_eo + n_el + n_do + n_dl);
    CK(cudaMemcpy(buf, eo, n_eo, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(buf + n_eo, e_lse, n_el, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(buf + n_eo + n_el, dout, n_do, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(buf + n_eo + n_el + n_do, dlse, n_dl, cudaMemcpyDeviceToHost));
    FILE *o = fopen(argv[2], "wb");
    if (!o) return 1;
    fwrite(&flags, 4, 1, o);
    fwrite(buf, 1, n_eo + n_el + n_do + n_dl, o);
    fclose(o);
    printf("c caller ok, status 0x%x\n", flags);
    return 0;
}
"""


def _compiler():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def _u16(t):
    return t.contiguous().view(torch.int16).numpy().astype(np.int16).tobytes()


def _i32(t):
    return np.ascontiguousarray(t.numpy().astype(np.int32)).tobytes()


def test_c_program_store_extend_decode(tmp_path):
    lib = cuda_build.build()
    w = W.make_workload("ccall", 40, 8, 128, 16, seed=31, decode_seq_lens=[1, 300, 2049],
                        extend_prefix_lens=[0, 200], extend_ext_lens=[130, 77], device="cpu")
    k_new, v_new, loc = w.new_tokens()
    full_k, full_v = w.k_pool.clone(), w.v_pool.clone()
    # the pool rows the store must write start as zeros in the file the program reads
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    kp[loc.long()] = 0
    vp[loc.long()] = 0
    e, d = w.extend, w.decode
    hdr = np.array([w.num_slots, w.page_size, w.hkv, w.hq, loc.numel(), e.num_reqs, e.total_tokens, d.num_reqs,
                    e.page_table.shape[1], d.page_table.shape[1]], dtype=np.int32)
    lim = np.array([e.max_ext_len, e.max_seq_len, d.max_seq_len, 0], dtype=np.int32)
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(hdr.tobytes())
        f.write(np.array([w.scale], dtype=np.float32).tobytes())
        f.write(lim.tobytes())
        for blob in (_u16(kp), _u16(vp), _u16(k_new), _u16(v_new), _i32(loc), _u16(e.q), _i32(e.page_table),
                     _i32(e.prefix_lens), _i32(e.ext_lens), _i32(e.cu_ext), _i32(e.positions), _u16(d.q),
                     _i32(d.page_table), _i32(d.seq_lens)):
            f.write(blob)
    src = tmp_path / "caller.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib)
    subprocess.run([_compiler(), "-x", "c", str(src), "-o", str(exe), "-I", os.path.join(ROOT, "include"),
                    "-L", libdir, "-lmsgl_attn", "-Xlinker", f"-rpath={libdir}"], check=True)
    out = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(inp), str(out)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = out.read_bytes()
    flags = np.frombuffer(raw[:4], dtype=np.uint32)[0]
    assert flags == 0
    T, B, hq = e.total_tokens, d.num_reqs, w.hq
    off = 4
    sizes = [T * hq * 256, T * hq * 4, B * hq * 256, B * hq * 4]
    parts = []
    for n in sizes:
        parts.append(raw[off:off + n])
        off += n
    bf = lambda b, shape: torch.from_numpy(np.frombuffer(b, dtype=np.int16).copy()).view(torch.bfloat16).reshape(shape)
    eo, el = bf(parts[0], (T, hq, 128)), np.frombuffer(parts[1], dtype=np.float32).reshape(T, hq)
    do, dl = bf(parts[2], (B, hq, 128)), np.frombuffer(parts[3], dtype=np.float32).reshape(B, hq)
    ref_o, ref_l = oracle.extend(e.q, full_k, full_v, w.page_size, e.page_table, e.prefix_lens, e.ext_lens, w.scale)
    a, _ = oracle.extend(e.q, full_k, full_v.abs(), w.page_size, e.page_table, e.prefix_lens, e.ext_lens, w.scale)
    assert_o_close(eo, ref_o, "C caller extend", abs_ref=a)
    assert_lse_close(el, ref_l, "C caller extend")
    ref_o, ref_l = oracle.decode(d.q, full_k, full_v, w.page_size, d.page_table, d.seq_lens, w.scale)
    a, _ = oracle.decode(d.q, full_k, full_v.abs(), w.page_size, d.page_table, d.seq_lens, w.scale)
    assert_o_close(do, ref_o, "C caller decode", abs_ref=a)
    assert_lse_close(dl, ref_l, "C caller decode")
