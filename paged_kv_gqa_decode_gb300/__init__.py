"""GB300 (sm_103a) paged-KV GQA decode attention.

A thin Python binding over the C ABI in ``include/paged_attn.h``: the
functions here only marshal torch tensors into pointers, sizes and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the compiled library is missing the
calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "PagedAttnError",
    "LIB_PATH",
    "load",
    "paged_attn_decode",
    "paged_attn_decode_ws",
    "paged_attn_decode_checked",
    "paged_attn_decode_static",
    "paged_attn_append_decode",
    "paged_kv_append",
    "paged_attn_decode_fp8",
    "paged_attn_decode_xpacked",
    "paged_attn_decode_multi",
    "paged_kv_append_multi",
    "paged_attn_append_decode_multi",
    "paged_kv_append_fp8",
    "paged_attn_append_decode_fp8",
    "paged_attn_workspace_bytes",
    "paged_attn_status_string",
    "paged_attn_set_launch_flags",
    "paged_attn_set_checks",
    "paged_attn_reset_workspace",
    "FLAG_EARLY_PROLOGUE",
    "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libpaged_kv_gqa_decode.so")

# Every symbol declared in include/paged_attn.h.
EXPORTED_SYMBOLS = (
    "paged_attn_decode",
    "paged_attn_workspace_bytes",
    "paged_attn_decode_ws",
    "paged_attn_decode_checked",
    "paged_attn_decode_static",
    "paged_kv_append",
    "paged_attn_append_decode",
    "paged_attn_decode_fp8",
    "paged_attn_decode_xpacked",
    "paged_attn_decode_multi",
    "paged_attn_decode_multi_ex",
    "paged_kv_append_multi",
    "paged_attn_append_decode_multi",
    "paged_kv_append_fp8",
    "paged_attn_append_decode_fp8",
    "paged_attn_status_string",
    "paged_attn_set_launch_flags",
    "paged_attn_set_checks",
    "paged_attn_reset_workspace",
    "paged_attn_last_cuda_error",
    "paged_attn_version",
)

# Launch flags (include/paged_attn.h).
FLAG_EARLY_PROLOGUE = 1

_lock = threading.Lock()
_lib = None


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"paged_attn status {status}: {message}")
        self.status = status


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the compiled library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with `python -m paged_kv_gqa_decode_gb300.build` "
                "(needs nvcc from the CUDA 13 toolkit)")
        lib = ctypes.CDLL(p)
        P, I, F, LL, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong,
                           ctypes.c_size_t)
        common = [P, P, P, P, P, P, I, I, I, I, I, I, F]
        lib.paged_attn_decode.argtypes = common + [P]
        lib.paged_attn_decode.restype = I
        lib.paged_attn_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.paged_attn_workspace_bytes.restype = SZ
        lib.paged_attn_decode_ws.argtypes = common + [P, SZ, P]
        lib.paged_attn_decode_ws.restype = I
        lib.paged_attn_decode_checked.argtypes = common + [LL, P, P]
        lib.paged_attn_decode_checked.restype = I
        lib.paged_attn_decode_static.argtypes = common + [P]
        lib.paged_attn_decode_static.restype = I
        lib.paged_kv_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P]
        lib.paged_kv_append.restype = I
        lib.paged_attn_append_decode.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.paged_attn_append_decode.restype = I
        lib.paged_attn_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.paged_attn_decode_fp8.restype = I
        lib.paged_attn_decode_xpacked.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.paged_attn_decode_xpacked.restype = I
        lib.paged_attn_decode_multi.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F,
                                                P]
        lib.paged_attn_decode_multi.restype = I
        lib.paged_attn_decode_multi_ex.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I,
                                                   F, I, P]
        lib.paged_attn_decode_multi_ex.restype = I
        lib.paged_kv_append_multi.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P]
        lib.paged_kv_append_multi.restype = I
        lib.paged_attn_append_decode_multi.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                                       I, I, I, F, I, P]
        lib.paged_attn_append_decode_multi.restype = I
        lib.paged_kv_append_fp8.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P]
        lib.paged_kv_append_fp8.restype = I
        lib.paged_attn_append_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I,
                                                     I, F, P]
        lib.paged_attn_append_decode_fp8.restype = I
        lib.paged_attn_set_checks.argtypes = [LL, P]
        lib.paged_attn_set_checks.restype = I
        lib.paged_attn_reset_workspace.argtypes = [P]
        lib.paged_attn_reset_workspace.restype = I
        lib.paged_attn_status_string.argtypes = [I]
        lib.paged_attn_status_string.restype = ctypes.c_char_p
        lib.paged_attn_last_cuda_error.argtypes = []
        lib.paged_attn_last_cuda_error.restype = I
        lib.paged_attn_version.argtypes = []
        lib.paged_attn_version.restype = I
        lib.paged_attn_set_launch_flags.argtypes = [I]
        lib.paged_attn_set_launch_flags.restype = I
        if path is None:
            _lib = lib
        return lib


def paged_attn_status_string(status: int) -> str:
    return load().paged_attn_status_string(int(status)).decode()


def paged_attn_set_launch_flags(flags: int) -> None:
    """Launch flags for later decode calls from this host thread (0: the plain
    launch).  FLAG_EARLY_PROLOGUE: the caller guarantees that the work ahead in
    the stream writes none of the caches, block tables, lengths or query offsets
    (see include/paged_attn.h).  paged_kv_append and paged_attn_append_decode
    write the cache, so a launch right after one of them on the same cache must
    not use it."""
    _check(load().paged_attn_set_launch_flags(int(flags)))


def paged_attn_set_checks(num_blocks: int = 0, status=None) -> None:
    """Device-side checks for later calls from this host thread: block ids are
    validated against [0, num_blocks) and problems reported into ``status`` (an
    int32 device tensor of one element the caller zero-fills); ``(0, None)``
    turns them off (see include/paged_attn.h)."""
    _check(load().paged_attn_set_checks(int(num_blocks), _ptr(status)))


def paged_attn_reset_workspace(stream=None) -> None:
    """Zero-fill the library-owned workspace of the current device (needed only
    after a call reported a combine wait that ran out)."""
    _check(load().paged_attn_reset_workspace(_stream(stream)))


def _check(status: int) -> None:
    if status != 0:
        lib = load()
        msg = lib.paged_attn_status_string(status).decode()
        if status == -6:
            msg += f" (CUDA error {lib.paged_attn_last_cuda_error()})"
        raise PagedAttnError(status, msg)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _sizes(q, k_cache, block_tables):
    num_seqs, H_q, D = (int(x) for x in q.shape)
    _, H_kv, BS, Dk = (int(x) for x in k_cache.shape)
    if Dk != D:
        raise ValueError("q and the caches disagree on head_dim")
    maxb = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    return num_seqs, H_q, H_kv, D, maxb, BS


def _args(q, k_cache, v_cache, out, block_tables, seq_lens, scale):
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out),
                    ("block_tables", block_tables), ("seq_lens", seq_lens)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    num_seqs, H_q, H_kv, D, maxb, BS = _sizes(q, k_cache, block_tables)
    return (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(block_tables),
            _ptr(seq_lens), num_seqs, H_q, H_kv, D, maxb, BS, float(scale))


def paged_attn_decode(q, k_cache, v_cache, block_tables, seq_lens, scale: float, out=None,
                      stream=None):
    """out[s, h] = softmax(scale * q[s, h] . K^T) . V over the paged cache (see paged_attn.h)."""
    import torch

    if out is None:
        out = torch.empty_like(q)
    _check(load().paged_attn_decode(*_args(q, k_cache, v_cache, out, block_tables, seq_lens,
                                           scale), _stream(stream)))
    return out


def paged_attn_workspace_bytes(num_seqs: int, H_q: int, H_kv: int, head_dim: int,
                               max_blocks_per_seq: int, block_size: int) -> int:
    return int(load().paged_attn_workspace_bytes(num_seqs, H_q, H_kv, head_dim,
                                                 max_blocks_per_seq, block_size))


def paged_attn_decode_ws(q, k_cache, v_cache, block_tables, seq_lens, scale: float, workspace,
                         out=None, stream=None):
    """As paged_attn_decode, with a caller-owned zero-initialised uint8 device workspace."""
    import torch

    if out is None:
        out = torch.empty_like(q)
    _check(load().paged_attn_decode_ws(*_args(q, k_cache, v_cache, out, block_tables, seq_lens,
                                              scale), _ptr(workspace),
                                       int(workspace.numel() * workspace.element_size()),
                                       _stream(stream)))
    return out


def paged_attn_decode_checked(q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                              status, out=None, stream=None, num_blocks: Optional[int] = None):
    """As paged_attn_decode, validating block ids and lengths on the device into ``status``
    (an int32 device tensor of one element that the caller zero-fills)."""
    import torch

    if out is None:
        out = torch.empty_like(q)
    nb = int(k_cache.shape[0]) if num_blocks is None else int(num_blocks)
    _check(load().paged_attn_decode_checked(*_args(q, k_cache, v_cache, out, block_tables,
                                                   seq_lens, scale), nb, _ptr(status),
                                            _stream(stream)))
    return out


def paged_attn_decode_static(q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                             out=None, stream=None):
    """As paged_attn_decode, for callers that must not allocate device memory: the
    library's fixed 4 MiB scratch array stands in for the workspace (see paged_attn.h;
    calls that overlap on the GPU race on that array).  ``out`` should be passed in by
    such callers, since creating it here would allocate."""
    import torch

    if out is None:
        out = torch.empty_like(q)
    _check(load().paged_attn_decode_static(*_args(q, k_cache, v_cache, out, block_tables,
                                                  seq_lens, scale), _stream(stream)))
    return out


def paged_attn_decode_xpacked(q, kx, vt, block_tables, seq_lens, scale: float, out=None,
                              stream=None):
    """Decode over x-packed bf16 caches (see paged_attn.h): kx [num_blocks, H_kv,
    head_dim / 8, block_size, 8], vt [num_blocks, H_kv, head_dim, block_size]."""
    import torch

    for name, t in (("q", q), ("kx", kx), ("vt", vt), ("block_tables", block_tables),
                    ("seq_lens", seq_lens)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    num_seqs, H_q, D = (int(x) for x in q.shape)
    if kx.dim() != 5 or vt.dim() != 4:
        raise ValueError("kx must be [NB, H_kv, D/8, BS, 8] and vt [NB, H_kv, D, BS]")
    nb, H_kv, dx, BS, x = (int(v) for v in kx.shape)
    if x != 8 or dx * 8 != D or tuple(vt.shape) != (nb, H_kv, D, BS):
        raise ValueError("kx / vt shapes do not match q's head_dim")
    if out is None:
        out = torch.empty_like(q)
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    maxb = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    _check(load().paged_attn_decode_xpacked(_ptr(q), _ptr(kx), _ptr(vt), _ptr(out),
                                            _ptr(block_tables), _ptr(seq_lens), num_seqs, H_q,
                                            H_kv, D, maxb, BS, float(scale), _stream(stream)))
    return out


def _multi_sizes(q, k_cache, qo_indptr, block_tables, seq_lens, contiguous):
    import torch

    for name, t in contiguous.items():
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    total_q, H_q, D = (int(x) for x in q.shape)
    _, H_kv, BS, Dk = (int(x) for x in k_cache.shape)
    if Dk != D:
        raise ValueError("q and the caches disagree on head_dim")
    num_seqs = int(seq_lens.shape[0])
    if tuple(qo_indptr.shape) != (num_seqs + 1,) or qo_indptr.dtype != torch.int32:
        raise ValueError("qo_indptr must be int32 [num_seqs + 1]")
    maxb = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    return num_seqs, total_q, H_q, H_kv, D, maxb, BS


def paged_attn_decode_multi(q, k_cache, v_cache, qo_indptr, block_tables, seq_lens,
                            scale: float, max_q_len: int, out=None, stream=None,
                            causal: bool = True):
    """Multi-token decode (see paged_attn.h): q [total_q, H_q, D], sequence s owning
    rows qo_indptr[s] .. qo_indptr[s+1] - 1 (its last tokens); causal, or every
    row attending all of the sequence's tokens with ``causal=False``."""
    import torch

    num_seqs, total_q, H_q, H_kv, D, maxb, BS = _multi_sizes(
        q, k_cache, qo_indptr, block_tables, seq_lens,
        dict(q=q, k_cache=k_cache, v_cache=v_cache, qo_indptr=qo_indptr,
             block_tables=block_tables, seq_lens=seq_lens))
    if out is None:
        out = torch.empty_like(q)
    _check(load().paged_attn_decode_multi_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                             _ptr(qo_indptr), _ptr(block_tables),
                                             _ptr(seq_lens), num_seqs, total_q, int(max_q_len),
                                             H_q, H_kv, D, maxb, BS, float(scale),
                                             1 if causal else 0, _stream(stream)))
    return out


def paged_kv_append_multi(k_new, v_new, k_cache, v_cache, qo_indptr, block_tables, seq_lens,
                          stream=None):
    """Write several new tokens per sequence into the paged caches (see paged_attn.h):
    k_new, v_new [total_q, H_kv, head_dim] bf16, row qo_indptr[s] + i being token
    seq_lens[s] - q_len + i of sequence s."""
    _check_rows(k_new, v_new, None, k_cache)
    num_seqs, total_q, _, H_kv, D, maxb, BS = _multi_sizes(
        k_new, k_cache, qo_indptr, block_tables, seq_lens,
        dict(qo_indptr=qo_indptr, block_tables=block_tables, seq_lens=seq_lens))
    _check(load().paged_kv_append_multi(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(qo_indptr), _ptr(block_tables), _ptr(seq_lens),
                                        num_seqs, total_q, H_kv, D, maxb, BS, _stream(stream)))


def paged_attn_append_decode_multi(q, k_new, v_new, k_cache, v_cache, qo_indptr, block_tables,
                                   seq_lens, scale: float, max_q_len: int, out=None,
                                   stream=None, causal: bool = True):
    """paged_kv_append_multi then paged_attn_decode_multi (see paged_attn.h)."""
    import torch

    _check_rows(k_new, v_new, q, k_cache)
    num_seqs, total_q, H_q, H_kv, D, maxb, BS = _multi_sizes(
        q, k_cache, qo_indptr, block_tables, seq_lens,
        dict(q=q, k_cache=k_cache, v_cache=v_cache, qo_indptr=qo_indptr,
             block_tables=block_tables, seq_lens=seq_lens))
    if out is None:
        out = torch.empty_like(q)
    _check(load().paged_attn_append_decode_multi(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(out),
        _ptr(qo_indptr), _ptr(block_tables), _ptr(seq_lens), num_seqs, total_q, int(max_q_len),
        H_q, H_kv, D, maxb, BS, float(scale), 1 if causal else 0, _stream(stream)))
    return out


def _check_rows(k_new, v_new, q_or_none, k_cache):
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _, H_kv, _, D = (int(x) for x in k_cache.shape)
    if tuple(k_new.shape[1:]) != (H_kv, D) or k_new.shape != v_new.shape:
        raise ValueError("k_new and v_new must be [num_seqs, H_kv, head_dim]")
    if q_or_none is not None and int(k_new.shape[0]) != int(q_or_none.shape[0]):
        raise ValueError("k_new must have one row set per sequence of q")


def paged_kv_append(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, stream=None):
    """Write each sequence's new token (position seq_lens[s] - 1) into the paged caches
    (see paged_attn.h).  k_new, v_new: [num_seqs, H_kv, head_dim] bf16."""
    _check_rows(k_new, v_new, None, k_cache)
    num_blocks, H_kv, BS, D = (int(x) for x in k_cache.shape)
    maxb = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    _check(load().paged_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_tables), _ptr(seq_lens), int(k_new.shape[0]), H_kv,
                                  D, maxb, BS, _stream(stream)))


def paged_attn_append_decode(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                             scale: float, out=None, stream=None):
    """paged_kv_append then paged_attn_decode, fused into one launch (see paged_attn.h)."""
    import torch

    _check_rows(k_new, v_new, q, k_cache)
    if out is None:
        out = torch.empty_like(q)
    a = _args(q, k_cache, v_cache, out, block_tables, seq_lens, scale)
    # (q, k_new, v_new, k_cache, v_cache, out, tables, lens, sizes..., scale)
    _check(load().paged_attn_append_decode(a[0], _ptr(k_new), _ptr(v_new), a[1], a[2], a[3],
                                           *a[4:], _stream(stream)))
    return out


def paged_attn_decode_fp8(q, k8, v8, k_scale, v_scale, block_tables, seq_lens, scale: float,
                          out=None, stream=None):
    """Decode over FP8 caches (see paged_attn.h): k8 / v8 hold e4m3 bytes (uint8)
    [num_blocks, H_kv, block_size, head_dim], k_scale / v_scale one float32 per
    (block, KV head, slot); head_dim 128 or 256."""
    import torch

    for name, t in (("k8", k8), ("v8", v8), ("k_scale", k_scale), ("v_scale", v_scale)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if k8.dtype != torch.uint8 or v8.dtype != torch.uint8:
        raise ValueError("k8 / v8 must be uint8 (e4m3 bytes)")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32 or \
            tuple(k_scale.shape) != tuple(k8.shape[:3]) or k_scale.shape != v_scale.shape:
        raise ValueError("k_scale / v_scale must be float32 [num_blocks, H_kv, block_size]")
    if out is None:
        out = torch.empty_like(q)
    a = _args(q, k8, v8, out, block_tables, seq_lens, scale)
    # (q, k8, v8, k_scale, v_scale, out, tables, lens, sizes..., scale)
    _check(load().paged_attn_decode_fp8(a[0], a[1], a[2], _ptr(k_scale), _ptr(v_scale), a[3],
                                        *a[4:], _stream(stream)))
    return out


def _check_fp8_cache(k8, v8, k_scale, v_scale):
    import torch

    for name, t in (("k8", k8), ("v8", v8), ("k_scale", k_scale), ("v_scale", v_scale)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if k8.dtype != torch.uint8 or v8.dtype != torch.uint8:
        raise ValueError("k8 / v8 must be uint8 (e4m3 bytes)")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32 or \
            tuple(k_scale.shape) != tuple(k8.shape[:3]) or k_scale.shape != v_scale.shape:
        raise ValueError("k_scale / v_scale must be float32 [num_blocks, H_kv, block_size]")


def paged_kv_append_fp8(k_new, v_new, k8, v8, k_scale, v_scale, block_tables, seq_lens,
                        stream=None):
    """Quantize each sequence's new K / V rows (bf16 [num_seqs, H_kv, head_dim]) to
    e4m3 with one dequant float per row and write them into the FP8 caches at
    position seq_lens[s] - 1 (see paged_attn.h)."""
    _check_fp8_cache(k8, v8, k_scale, v_scale)
    _check_rows(k_new, v_new, None, k8)
    num_blocks, H_kv, BS, D = (int(x) for x in k8.shape)
    maxb = int(block_tables.shape[1]) if block_tables.dim() == 2 else 0
    _check(load().paged_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k8), _ptr(v8),
                                      _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                      _ptr(seq_lens), int(k_new.shape[0]), H_kv, D, maxb, BS,
                                      _stream(stream)))


def paged_attn_append_decode_fp8(q, k_new, v_new, k8, v8, k_scale, v_scale, block_tables,
                                 seq_lens, scale: float, out=None, stream=None):
    """paged_kv_append_fp8 then paged_attn_decode_fp8 (see paged_attn.h)."""
    import torch

    _check_fp8_cache(k8, v8, k_scale, v_scale)
    _check_rows(k_new, v_new, q, k8)
    if out is None:
        out = torch.empty_like(q)
    a = _args(q, k8, v8, out, block_tables, seq_lens, scale)
    # (q, k_new, v_new, k8, v8, k_scale, v_scale, out, tables, lens, sizes..., scale)
    _check(load().paged_attn_append_decode_fp8(a[0], _ptr(k_new), _ptr(v_new), a[1], a[2],
                                               _ptr(k_scale), _ptr(v_scale), a[3], *a[4:],
                                               _stream(stream)))
    return out
