"""fp64 CPU oracle for paged grouped-query attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference`` arm) may import this package.
The CUDA library never imports, links or calls it, and it imports nothing
from the CUDA library: the two share no code.  Inputs reach both sides from
the seeded generators in ``paged_kv_attention_24_gb300.workloads`` (which
hold none of the method's arithmetic).

The arithmetic lives in ``msgl_oracle.c`` (plain C, fp64); this module
compiles it with gcc on first use and marshals arrays through ctypes.
What it computes, term by term, is written at the top of that file; the
passages it follows are:

* unified KV pool, page as its allocation unit, configurable page size:
  "Mini-SGLang 实战指南", §6.2 "Page Size", §6.5 "Radix Cache";
* attention metadata (page table, positions) and "KV = pool history + newly
  computed KV": "不懂SGLang？从miniSGLang开始", §1.3 "前向运算";
* a prefill chunk attends over the cached prefix plus itself causally:
  "Mini-SGLang 实战指南", §6.1 "Chunked Prefill";
* prefill and decode as separate attention calls: "Mini-SGLang 实战指南",
  §6.3.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msgl_oracle.c")
_lock = threading.Lock()
_libs: dict = {}


def build(mutant: int = 0, out_dir: str | None = None) -> str:
    """Compile the oracle (optionally a planted-mistake variant); return the .so path."""
    out_dir = out_dir or os.path.join(_HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    name = "libmsgl_oracle.so" if mutant == 0 else f"libmsgl_oracle_mutant{mutant}.so"
    out = os.path.join(out_dir, name)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-shared", "-fPIC",
           "-pthread", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutant: int = 0):
    with _lock:
        if mutant not in _libs:
            lib = ctypes.CDLL(build(mutant))
            P = ctypes.c_void_p
            lib.oracle_store_kv.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                            P, P, P, ctypes.c_int64]
            lib.oracle_store_kv.restype = ctypes.c_int
            lib.oracle_attention_items.argtypes = [
                P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int64,
                ctypes.c_int32, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
                ctypes.c_int64, P, P, P, P, P, P, ctypes.c_int32]
            lib.oracle_attention_items.restype = ctypes.c_int
            lib.oracle_mutant_id.restype = ctypes.c_int
            _libs[mutant] = lib
        return _libs[mutant]


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 numpy array of bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16, x.dtype
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def store_kv(k_pool, v_pool, k_new, v_new, out_loc, mutant: int = 0):
    """Scatter new K/V rows into copies of the pools; returns (k_pool, v_pool) as uint16 bits.

    k_pool/v_pool: [S, Hkv, D] bf16 (or uint16 bits); k_new/v_new: [N, Hkv, D]; out_loc: [N].
    """
    kp = _bits(k_pool).copy()
    vp = _bits(v_pool).copy()
    kn, vn, loc = _bits(k_new), _bits(v_new), _i32(out_loc)
    S, hkv, d = kp.shape
    n = loc.shape[0]
    assert kn.shape == (n, hkv, d) and vn.shape == (n, hkv, d)
    rc = _lib(mutant).oracle_store_kv(_ptr(kp), _ptr(vp), S, hkv, d, _ptr(kn), _ptr(vn), _ptr(loc), n)
    if rc:
        raise OracleError(f"oracle_store_kv failed with status {rc}")
    return kp, vp


def attention_items(q, k_pool, v_pool, page_size, page_table, scale, item_req, item_qrow,
                    item_pos, item_head, n_threads: int | None = None, mutant: int = 0):
    """Attention for explicit (request, q row, absolute position, q head) items.

    Returns (o [n, D] fp64, lse [n] fp64).  ``page_table`` is [B, W] int32 of page ids.
    """
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    pt = _i32(page_table)
    if pt.ndim == 1:
        pt = pt.reshape(1, -1)
    S, hkv, d = kb.shape
    hq = qb.shape[1]
    assert qb.shape[2] == d and vb.shape == kb.shape
    req, qrow, pos, head = (_i32(item_req), _i32(item_qrow), _i32(item_pos), _i32(item_head))
    n = req.shape[0]
    assert qrow.shape[0] == n and pos.shape[0] == n and head.shape[0] == n
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    if n == 0:
        return o, lse
    rc = _lib(mutant).oracle_attention_items(
        _ptr(qb), hq, hkv, d, _ptr(kb), _ptr(vb), S, int(page_size), _ptr(pt), pt.shape[1],
        pt.shape[1], float(scale), n, _ptr(req), _ptr(qrow), _ptr(pos), _ptr(head),
        _ptr(o), _ptr(lse), int(n_threads or default_threads()))
    if rc:
        raise OracleError(f"oracle_attention_items failed with status {rc}")
    return o, lse


def extend(q, k_pool, v_pool, page_size, page_table, prefix_lens, ext_lens, scale,
           n_threads: int | None = None, mutant: int = 0):
    """Chunked-prefill attention: row i of request b sits at position prefix_b + i.

    q: [T, Hq, D] (request-major, ext_lens rows per request).  Returns
    (o [T, Hq, D] fp64, lse [T, Hq] fp64).
    """
    pre, ext = _i32(prefix_lens), _i32(ext_lens)
    hq, d = q.shape[1], q.shape[2]
    T = int(ext.sum())
    assert q.shape[0] == T, (q.shape, T)
    reqs, rows, poss = [], [], []
    t = 0
    for b in range(pre.shape[0]):
        for i in range(int(ext[b])):
            reqs.append(b); rows.append(t); poss.append(int(pre[b]) + i)
            t += 1
    req = np.repeat(np.array(reqs, dtype=np.int32), hq)
    row = np.repeat(np.array(rows, dtype=np.int32), hq)
    pos = np.repeat(np.array(poss, dtype=np.int32), hq)
    head = np.tile(np.arange(hq, dtype=np.int32), T)
    o, lse = attention_items(q, k_pool, v_pool, page_size, page_table, scale, req, row, pos, head,
                             n_threads=n_threads, mutant=mutant)
    return o.reshape(T, hq, d), lse.reshape(T, hq)


def decode(q, k_pool, v_pool, page_size, page_table, seq_lens, scale,
           n_threads: int | None = None, mutant: int = 0):
    """One query row per request at position seq_b - 1 (it attends all seq_b keys).

    q: [B, Hq, D].  Returns (o [B, Hq, D] fp64, lse [B, Hq] fp64).
    """
    seq = _i32(seq_lens)
    B, hq, d = q.shape
    req = np.repeat(np.arange(B, dtype=np.int32), hq)
    pos = np.repeat(seq - 1, hq).astype(np.int32)
    head = np.tile(np.arange(hq, dtype=np.int32), B)
    o, lse = attention_items(q, k_pool, v_pool, page_size, page_table, scale, req, req, pos, head,
                             n_threads=n_threads, mutant=mutant)
    return o.reshape(B, hq, d), lse.reshape(B, hq)


def mutant_id(mutant: int) -> int:
    return int(_lib(mutant).oracle_mutant_id())
