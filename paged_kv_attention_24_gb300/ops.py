"""Thin ctypes binding over libmsgl_attn (argument marshalling only).

Every function here converts torch tensors to raw device pointers and host
scalars, calls the C ABI declared in ``include/msgl_attn.h`` with the
current CUDA stream, and turns a non-OK status into :class:`MsglError`.
All compute happens in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and calling anything here without the built library
raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libmsgl_attn.so")

MSGL_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "OUT_OF_RANGE",
                5: "TIMEOUT", 6: "WORKSPACE"}
DEVERR_SLOT_RANGE = 0x1
DEVERR_PAGE_RANGE = 0x2
DEVERR_LENGTH = 0x4
DEVERR_POSITION = 0x8
DEVERR_TIMEOUT = 0x10
DEVERR_APPEND_SLOT = 0x20


class MsglError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"msgl status {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Pool(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_slots", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class _Pages(ctypes.Structure):
    _fields_ = [("page_ids", ctypes.c_void_p), ("stride", ctypes.c_int32),
                ("width", ctypes.c_int32)]


class _ExtendBatch(ctypes.Structure):
    _fields_ = [("pages", _Pages), ("q", ctypes.c_void_p), ("prefix_lens", ctypes.c_void_p),
                ("ext_lens", ctypes.c_void_p), ("cu_ext", ctypes.c_void_p), ("positions", ctypes.c_void_p),
                ("num_reqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("max_ext_len", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class _DecodeBatch(ctypes.Structure):
    _fields_ = [("pages", _Pages), ("q", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("num_reqs", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()

P, I32, I64, SZ, F32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                        ctypes.c_float)
PP = ctypes.POINTER(_Pool)
PT = ctypes.POINTER(_Pages)

SIGNATURES = {
    "msgl_store_kv": ([PP, P, P, P, I32, P, P], ctypes.c_int),
    "msgl_extend_workspace_size": ([I32, I32, I32, I32, I32, I32], SZ),
    "msgl_attn_extend": ([PP, PT, P, I32, P, P, P, P, I32, I32, I32, I32, F32, P, P, P, SZ, P, P],
                         ctypes.c_int),
    "msgl_decode_workspace_size": ([I32, I32, I32, I32, I32], SZ),
    "msgl_attn_decode": ([PP, PT, P, I32, P, I32, I32, F32, P, P, P, SZ, P, P], ctypes.c_int),
    "msgl_attn_decode_append": ([PP, PT, P, I32, P, P, P, P, I32, I32, F32, P, P, P, SZ, P, P], ctypes.c_int),
    "msgl_attn_decode_noalloc": ([PP, PT, P, I32, P, I32, I32, F32, P, P, P, P], ctypes.c_int),
    "msgl_attn_mixed": ([PP, ctypes.POINTER(_ExtendBatch), ctypes.POINTER(_DecodeBatch), I32, F32, P, SZ, P, P],
                        ctypes.c_int),
    "msgl_selftest_wait_timeout": ([P, I64, P], ctypes.c_int),
    "msgl_read_status": ([P, ctypes.POINTER(ctypes.c_uint32), P], ctypes.c_int),
    "msgl_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "msgl_last_error": ([], ctypes.c_char_p),
    "msgl_abi_version": ([], I32),
    "msgl_check_store_meta": ([I64, P, I32], ctypes.c_int),
    "msgl_check_extend_meta": ([I64, I32, P, I32, I32, P, P, P, P, I32, I32, I32, I32], ctypes.c_int),
    "msgl_check_decode_meta": ([I64, I32, P, I32, I32, P, I32, I32], ctypes.c_int),
}


def load(path: Optional[str] = None):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libmsgl_attn is not built ({p} missing); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        if path is None:
            _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != MSGL_OK:
        msg = load().msgl_last_error().decode(errors="replace")
        raise MsglError(rc, f"{what}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class KVPool:
    """A layer's unified KV pool: bf16 K and V tensors [num_slots, Hkv, 128]."""

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor, page_size: int):
        _need(k_pool, "k_pool", torch.bfloat16)
        _need(v_pool, "v_pool", torch.bfloat16)
        if k_pool.shape != v_pool.shape or k_pool.dim() != 3:
            raise ValueError("k_pool and v_pool must both be [num_slots, Hkv, D]")
        self.k, self.v, self.page_size = k_pool, v_pool, int(page_size)

    @property
    def num_kv_heads(self) -> int:
        return int(self.k.shape[1])

    def c(self) -> _Pool:
        return _Pool(self.k.data_ptr(), self.v.data_ptr(), self.k.shape[0], self.page_size,
                     self.k.shape[1], self.k.shape[2])


def _pages(page_table: torch.Tensor) -> _Pages:
    _need(page_table, "page_table", torch.int32)
    if page_table.dim() != 2:
        raise ValueError("page_table must be [num_reqs, width]")
    return _Pages(page_table.data_ptr(), page_table.shape[1], page_table.shape[1])


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def store_kv(pool: KVPool, k: torch.Tensor, v: torch.Tensor, out_loc: torch.Tensor,
             status: Optional[torch.Tensor] = None, stream=None) -> None:
    """pool.k[out_loc[t]] = k[t]; pool.v[out_loc[t]] = v[t] (bit-exact)."""
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    _need(out_loc, "out_loc", torch.int32)
    pc = pool.c()
    rc = load().msgl_store_kv(ctypes.byref(pc), _ptr(k), _ptr(v), _ptr(out_loc), int(out_loc.shape[0]),
                              _ptr(status), _stream(stream))
    _check(rc, "msgl_store_kv")


def decode_workspace_size(num_reqs: int, hq: int, hkv: int, max_seq_len: int, head_dim: int = 128) -> int:
    return int(load().msgl_decode_workspace_size(num_reqs, hq, hkv, head_dim, max_seq_len))


def extend_workspace_size(num_reqs: int, total_tokens: int, hq: int, hkv: int, max_seq_len: int,
                          head_dim: int = 128) -> int:
    return int(load().msgl_extend_workspace_size(num_reqs, total_tokens, hq, hkv, head_dim, max_seq_len))


def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def attn_decode(pool: KVPool, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                max_seq_len: int, scale: float, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None):
    """One query row per request over all its pages; returns (o bf16 [B,Hq,D], lse fp32 [B,Hq])."""
    _need(q, "q", torch.bfloat16)
    _need(seq_lens, "seq_lens", torch.int32)
    B, hq, d = q.shape
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, hq, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    if workspace is None:
        workspace = _workspace(decode_workspace_size(B, hq, pool.num_kv_heads, max_seq_len, d), q.device)
    pc, pt = pool.c(), _pages(page_table)
    rc = load().msgl_attn_decode(
        ctypes.byref(pc), ctypes.byref(pt), _ptr(q), hq, _ptr(seq_lens), B, int(max_seq_len),
        float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _check(rc, "msgl_attn_decode")
    return out, lse


def attn_extend(pool: KVPool, q: torch.Tensor, page_table: torch.Tensor, prefix_lens: torch.Tensor,
                ext_lens: torch.Tensor, cu_ext: torch.Tensor, max_ext_len: int, max_seq_len: int,
                scale: float, positions: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                stream=None):
    """Chunked prefill over cached prefix + causal chunk; returns (o [T,Hq,D], lse [T,Hq])."""
    _need(q, "q", torch.bfloat16)
    for name, t in (("prefix_lens", prefix_lens), ("ext_lens", ext_lens), ("cu_ext", cu_ext)):
        _need(t, name, torch.int32)
    if positions is not None:
        _need(positions, "positions", torch.int32)
    T, hq, d = q.shape
    B = int(prefix_lens.shape[0])
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(T, hq, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    if workspace is None:
        workspace = _workspace(extend_workspace_size(B, T, hq, pool.num_kv_heads, max_seq_len, d), q.device)
    pc, pt = pool.c(), _pages(page_table)
    rc = load().msgl_attn_extend(
        ctypes.byref(pc), ctypes.byref(pt), _ptr(q), hq, _ptr(prefix_lens), _ptr(ext_lens),
        _ptr(cu_ext), _ptr(positions), B, T, int(max_ext_len), int(max_seq_len), float(scale),
        _ptr(out), _ptr(lse), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _check(rc, "msgl_attn_extend")
    return out, lse


def attn_decode_append(pool: KVPool, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       new_loc: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                       max_seq_len: int, scale: float, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None, stream=None):
    """Store each request's current-token K/V at new_loc and decode, in one launch."""
    _need(q, "q", torch.bfloat16)
    _need(k_new, "k_new", torch.bfloat16)
    _need(v_new, "v_new", torch.bfloat16)
    _need(new_loc, "new_loc", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, hq, d = q.shape
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, hq, dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    if workspace is None:
        workspace = _workspace(decode_workspace_size(B, hq, pool.num_kv_heads, max_seq_len, d), q.device)
    pc, pt = pool.c(), _pages(page_table)
    rc = load().msgl_attn_decode_append(
        ctypes.byref(pc), ctypes.byref(pt), _ptr(q), hq, _ptr(k_new), _ptr(v_new), _ptr(new_loc),
        _ptr(seq_lens), B, int(max_seq_len), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(status),
        _stream(stream))
    _check(rc, "msgl_attn_decode_append")
    return out, lse


def attn_mixed(pool: KVPool, scale: float,
               ext_q: torch.Tensor, ext_page_table: torch.Tensor, prefix_lens: torch.Tensor,
               ext_lens: torch.Tensor, cu_ext: torch.Tensor, max_ext_len: int, max_ext_seq_len: int,
               dec_q: torch.Tensor, dec_page_table: torch.Tensor, seq_lens: torch.Tensor, max_dec_seq_len: int,
               positions: Optional[torch.Tensor] = None, ext_out=None, ext_lse=None, dec_out=None, dec_lse=None,
               workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None, stream=None):
    """The extend batch and the decode batch of one forward in one call (msgl_attn_mixed).

    Same results as :func:`attn_extend` and :func:`attn_decode`; returns
    ((o_ext, lse_ext), (o_dec, lse_dec)).
    """
    _need(ext_q, "ext_q", torch.bfloat16)
    _need(dec_q, "dec_q", torch.bfloat16)
    for name, t in (("prefix_lens", prefix_lens), ("ext_lens", ext_lens), ("cu_ext", cu_ext),
                    ("seq_lens", seq_lens)):
        _need(t, name, torch.int32)
    if positions is not None:
        _need(positions, "positions", torch.int32)
    T, hq, d = ext_q.shape
    B = int(dec_q.shape[0])
    if dec_q.shape[1] != hq:
        raise ValueError("ext_q and dec_q must have the same number of q heads")
    ext_out = torch.empty_like(ext_q) if ext_out is None else ext_out
    ext_lse = torch.empty(T, hq, dtype=torch.float32, device=ext_q.device) if ext_lse is None else ext_lse
    dec_out = torch.empty_like(dec_q) if dec_out is None else dec_out
    dec_lse = torch.empty(B, hq, dtype=torch.float32, device=dec_q.device) if dec_lse is None else dec_lse
    for name, t, dt in (("ext_out", ext_out, torch.bfloat16), ("ext_lse", ext_lse, torch.float32),
                        ("dec_out", dec_out, torch.bfloat16), ("dec_lse", dec_lse, torch.float32)):
        _need(t, name, dt)
    if workspace is None:
        workspace = _workspace(mixed_workspace_size(B, T, int(prefix_lens.shape[0]), hq, pool.num_kv_heads,
                                                    max_ext_seq_len, max_dec_seq_len, d), dec_q.device)
    eb = _ExtendBatch(_pages(ext_page_table), ext_q.data_ptr(), prefix_lens.data_ptr(), ext_lens.data_ptr(),
                      cu_ext.data_ptr(), None if positions is None else positions.data_ptr(),
                      int(prefix_lens.shape[0]), T, int(max_ext_len), int(max_ext_seq_len),
                      ext_out.data_ptr(), ext_lse.data_ptr())
    db = _DecodeBatch(_pages(dec_page_table), dec_q.data_ptr(), seq_lens.data_ptr(), B, int(max_dec_seq_len),
                      dec_out.data_ptr(), dec_lse.data_ptr())
    pc = pool.c()
    rc = load().msgl_attn_mixed(ctypes.byref(pc), ctypes.byref(eb), ctypes.byref(db), hq, float(scale),
                                _ptr(workspace),
                                0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _ptr(status), _stream(stream))
    _check(rc, "msgl_attn_mixed")
    return (ext_out, ext_lse), (dec_out, dec_lse)


def mixed_workspace_size(dec_reqs: int, ext_tokens: int, ext_reqs: int, hq: int, hkv: int,
                         max_ext_seq_len: int, max_dec_seq_len: int, head_dim: int = 128) -> int:
    """Workspace bytes of :func:`attn_mixed`: the decode's (rounded up to 256) plus the extend's."""
    dec = decode_workspace_size(dec_reqs, hq, hkv, max_dec_seq_len, head_dim) if dec_reqs > 0 else 0
    ext = extend_workspace_size(ext_reqs, ext_tokens, hq, hkv, max_ext_seq_len, head_dim) if ext_reqs > 0 else 0
    return (dec + 255) // 256 * 256 + ext


NOALLOC_SCRATCH_BYTES = 32 << 20


def attn_decode_noalloc(pool: KVPool, q: torch.Tensor, page_table: torch.Tensor,
                        seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                        out: torch.Tensor, lse: torch.Tensor,
                        status: Optional[torch.Tensor] = None, stream=None):
    """Decode with the library's built-in scratch instead of a workspace.

    For callers that must not allocate device memory: the caller passes the
    output buffers, and the library allocates nothing.  Same results as
    :func:`attn_decode`.
    """
    _need(q, "q", torch.bfloat16)
    _need(seq_lens, "seq_lens", torch.int32)
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    B, hq, _ = q.shape
    pc, pt = pool.c(), _pages(page_table)
    rc = load().msgl_attn_decode_noalloc(
        ctypes.byref(pc), ctypes.byref(pt), _ptr(q), hq, _ptr(seq_lens), B, int(max_seq_len),
        float(scale), _ptr(out), _ptr(lse), _ptr(status), _stream(stream))
    _check(rc, "msgl_attn_decode_noalloc")
    return out, lse


def selftest_wait_timeout(status: torch.Tensor, budget_cycles: int = 10_000_000, stream=None) -> None:
    """Run the bounded-wait self-test; the status word then holds DEVERR_TIMEOUT."""
    rc = load().msgl_selftest_wait_timeout(_ptr(status), int(budget_cycles), _stream(stream))
    _check(rc, "msgl_selftest_wait_timeout")


def read_status(status: torch.Tensor, stream=None) -> int:
    """Synchronise and return the device status word's bits (through the C ABI)."""
    flags = ctypes.c_uint32(0)
    rc = load().msgl_read_status(_ptr(status), ctypes.byref(flags), _stream(stream))
    if rc not in (0, 4, 5):
        _check(rc, "msgl_read_status")
    return int(flags.value)


# ------------------------------------------------------------ metadata checks (host)

def _host_i32(t):
    """A host int32 copy of a tensor (any device) or None, plus its ctypes pointer."""
    if t is None:
        return None, None
    a = t.detach().to("cpu", torch.int32).contiguous()
    return a, ctypes.c_void_p(a.data_ptr())


def check_store_meta(out_loc: torch.Tensor, num_slots: int):
    """Copies out_loc back and checks it: every slot in range, none twice.  Raises MsglError."""
    a, p = _host_i32(out_loc)
    _check(load().msgl_check_store_meta(int(num_slots), p, a.numel()), "msgl_check_store_meta")


def _table(page_table: torch.Tensor):
    a, p = _host_i32(page_table)
    if a.dim() == 1:
        a = a.reshape(1, -1)
    return a, p, int(a.shape[1])


def check_extend_meta(num_slots: int, page_size: int, page_table: torch.Tensor, prefix_lens: torch.Tensor,
                      ext_lens: torch.Tensor, cu_ext: torch.Tensor, positions: Optional[torch.Tensor],
                      max_ext_len: int, max_seq_len: int):
    """Copies an extend step's metadata back and checks it (lengths, positions, pages).  Raises MsglError."""
    pt, ptp, w = _table(page_table)
    pre, prep = _host_i32(prefix_lens)
    ext, extp = _host_i32(ext_lens)
    cu, cup = _host_i32(cu_ext)
    pos, posp = _host_i32(positions)
    if cu.numel() != pre.numel() + 1 or ext.numel() != pre.numel():
        raise ValueError("cu_ext must have num_reqs + 1 entries and ext_lens num_reqs")
    total = int(pos.numel()) if pos is not None else int(cu[-1])
    _check(load().msgl_check_extend_meta(int(num_slots), int(page_size), ptp, w, w, prep, extp, cup, posp,
                                         pre.numel(), total, int(max_ext_len), int(max_seq_len)),
           "msgl_check_extend_meta")


def check_decode_meta(num_slots: int, page_size: int, page_table: torch.Tensor, seq_lens: torch.Tensor,
                      max_seq_len: int):
    """Copies a decode step's metadata back and checks it (lengths, pages).  Raises MsglError."""
    pt, ptp, w = _table(page_table)
    seq, seqp = _host_i32(seq_lens)
    _check(load().msgl_check_decode_meta(int(num_slots), int(page_size), ptp, w, w, seqp, seq.numel(),
                                         int(max_seq_len)), "msgl_check_decode_meta")
