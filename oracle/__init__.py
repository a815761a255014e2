"""FP64 CPU oracle for single-token paged-KV GQA decode attention.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the product path never
imports this package, and this package imports nothing from it.

* ``decode``       -- the definition (plain two-pass softmax over the paged
                      layout) for every (s, h) row or for a list of rows; the C
                      source ``paged_attn_oracle.c`` states it in full.
* ``pieces``       -- the per-range softmax pieces (M, l, o) of rows.
* ``append``       -- the cache write of each sequence's new token (the step
                      before the decode); ``append_multi`` the write of several
                      new tokens per sequence along ``qo_indptr``.
* ``append_fp8``   -- the cache write into FP8 caches: each new row quantized
                      to e4m3 with its own dequant float (``quantize_rows_e4m3``;
                      ``e4m3_encode`` is the nearest-code rounding it uses).
* ``decode_fp8``   -- the definition over FP8 caches (e4m3 bytes and a dequant
                      float per cache row); ``e4m3_table`` decodes the 256
                      byte values from the format's bit fields.
* ``decode_xpacked`` -- the definition over x-packed K ([blocks, H_kv, D/8,
                      BS, 8]) and D-major V ([blocks, H_kv, D, BS]) caches.
* ``decode_multi`` -- several causal query tokens per sequence (rows through
                      ``qo_indptr``); query i of q_len sees t <= L - q_len + i.
* ``combine`` / ``finish`` -- the merge of two partial softmax states and the
                      final normalisation, as "Paged Attention Kernel
                      Architecture for BI-V100" (section 2, Level 1: the
                      ``attention_partial`` compound value and its binary
                      ``combine``) defines them, with an empty state (M = -inf)
                      contributing weight zero.

Pins (tests/test_oracle_pins.py) tie the oracle to a library routine
(torch's float64 scaled_dot_product_attention on the un-paged layout), closed
forms, invariances and a hand-derived golden example.

Parity unpinned: the zero row for a sequence with no tokens (L = 0), and for a
multi-token query that sees no token.  No page defines an empty softmax; the
oracle and the kernels implement the same reading.
"""
from __future__ import annotations

import copy
import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {
    0: "ok",
    -1: "invalid arguments",
    -2: "H_q is not a multiple of H_kv",
    -3: "a sequence length is negative or longer than max_blocks_per_seq * block_size",
    -4: "a block-table entry in use is outside [0, num_blocks)",
    -5: "out of host memory",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            LL = ctypes.c_longlong
            F = ctypes.c_float
            lib.oracle_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, LL, F, P, I]
            lib.oracle_decode.restype = I
            lib.oracle_decode_pairs.argtypes = [P, P, P, P, P, I, I, I, I, I, I, LL, F, P, I, P, I]
            lib.oracle_decode_pairs.restype = I
            lib.oracle_partial_pairs.argtypes = [P, P, P, P, P, I, I, I, I, I, I, LL, F, P, P, I,
                                                 P, P, P]
            lib.oracle_partial_pairs.restype = I
            lib.oracle_decode_fp8_pairs.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, LL, F,
                                                     P, I, P, I]
            lib.oracle_decode_fp8_pairs.restype = I
            lib.oracle_decode_xpacked_pairs.argtypes = [P, P, P, P, P, I, I, I, I, I, I, LL, F,
                                                         P, I, P, I]
            lib.oracle_decode_xpacked_pairs.restype = I
            lib.oracle_decode_multi.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, LL, F, I, P, I]
            lib.oracle_decode_multi.restype = I
            lib.oracle_e4m3_table.argtypes = [P]
            lib.oracle_e4m3_table.restype = None
            lib.oracle_e4m3_encode.argtypes = [P, I, P]
            lib.oracle_e4m3_encode.restype = None
            lib.oracle_quantize_rows_e4m3.argtypes = [P, I, I, P, P]
            lib.oracle_quantize_rows_e4m3.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = I
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _bits(x) -> np.ndarray:
    """bf16 data as a contiguous uint16 array (torch tensor or uint16 ndarray)."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch  # only for converting tensors handed in by the tests

    t = x.detach()
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.int32)
    return np.ascontiguousarray(x.detach().cpu().numpy(), dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Inputs:
    """Host views of one decode problem in the layout the oracle reads."""

    def __init__(self, q, k_cache, v_cache, block_tables, seq_lens, scale: float):
        self.q = _bits(q)
        self.k = _bits(k_cache)
        self.v = _bits(v_cache)
        self.bt = _i32(block_tables)
        self.lens = _i32(seq_lens)
        if self.q.ndim != 3 or self.k.ndim != 4 or self.k.shape != self.v.shape:
            raise ValueError("q must be [S,H_q,D] and the caches [NB,H_kv,BS,D]")
        self.num_seqs, self.H_q, self.D = self.q.shape
        self.num_blocks, self.H_kv, self.BS, Dk = self.k.shape
        if Dk != self.D:
            raise ValueError("head_dim of q and of the caches differ")
        if self.bt.ndim != 2 or self.bt.shape[0] != self.num_seqs:
            raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
        if self.lens.shape != (self.num_seqs,):
            raise ValueError("seq_lens must be [num_seqs]")
        self.maxb = self.bt.shape[1]
        self.scale = float(np.float32(scale))

    @classmethod
    def from_workload(cls, w) -> "Inputs":
        return cls(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)

    def _common(self):
        return (_ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.bt), _ptr(self.lens),
                self.num_seqs, self.H_q, self.H_kv, self.D, self.maxb, self.BS,
                self.num_blocks, self.scale)


def _as_inputs(x) -> Inputs:
    return x if isinstance(x, Inputs) else Inputs.from_workload(x)


def decode(x, pairs: Optional[Sequence[Sequence[int]]] = None, num_threads: int = 0) -> np.ndarray:
    """The definition in float64.

    ``x`` is a ``workloads.Workload`` or ``Inputs``.  Without ``pairs`` the
    result is ``[num_seqs, H_q, D]``; with ``pairs`` (a list of (s, h)) it is
    ``[len(pairs), D]``.
    """
    inp = _as_inputs(x)
    lib = _load()
    if pairs is None:
        out = np.zeros((inp.num_seqs, inp.H_q, inp.D), dtype=np.float64)
        rc = lib.oracle_decode(*inp._common(), _ptr(out), int(num_threads))
    else:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((pr.shape[0], inp.D), dtype=np.float64)
        rc = lib.oracle_decode_pairs(*inp._common(), _ptr(pr), pr.shape[0], _ptr(out),
                                     int(num_threads))
    if rc != 0:
        raise OracleError(f"oracle rejected the input: {ERRORS.get(rc, rc)}")
    return out


class Fp8Inputs:
    """Host views of one decode problem over FP8 caches: e4m3 bytes in the bf16
    layout plus one float per (block, KV head, slot) for K and for V."""

    def __init__(self, q, k8, v8, k_scale, v_scale, block_tables, seq_lens, scale: float):
        self.q = _bits(q)
        self.k8 = _u8(k8)
        self.v8 = _u8(v8)
        self.ks = _f32(k_scale)
        self.vs = _f32(v_scale)
        self.bt = _i32(block_tables)
        self.lens = _i32(seq_lens)
        if self.q.ndim != 3 or self.k8.ndim != 4 or self.k8.shape != self.v8.shape:
            raise ValueError("q must be [S,H_q,D] and the caches [NB,H_kv,BS,D]")
        self.num_seqs, self.H_q, self.D = self.q.shape
        self.num_blocks, self.H_kv, self.BS, Dk = self.k8.shape
        if Dk != self.D:
            raise ValueError("head_dim of q and of the caches differ")
        if self.ks.shape != self.k8.shape[:3] or self.vs.shape != self.ks.shape:
            raise ValueError("scales must be [NB, H_kv, BS]")
        self.maxb = self.bt.shape[1]
        self.scale = float(np.float32(scale))

    @classmethod
    def from_workload(cls, w) -> "Fp8Inputs":
        return cls(w.q, w.k8, w.v8, w.k_scale, w.v_scale, w.block_tables, w.seq_lens, w.scale)


def _u8(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.uint8)
    import torch

    return x.detach().cpu().contiguous().view(torch.uint8).numpy()


def _f32(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float32)
    return np.ascontiguousarray(x.detach().cpu().float().numpy(), dtype=np.float32)


def decode_fp8(x, pairs: Optional[Sequence[Sequence[int]]] = None,
               num_threads: int = 0) -> np.ndarray:
    """The definition over FP8 caches in float64: every K/V element is its e4m3
    value times the float of its (block, KV head, slot) row; see the C source."""
    inp = x if isinstance(x, Fp8Inputs) else Fp8Inputs.from_workload(x)
    if pairs is None:
        pr = np.stack(np.meshgrid(np.arange(inp.num_seqs), np.arange(inp.H_q), indexing="ij"),
                      axis=-1).reshape(-1, 2).astype(np.int32)
    else:
        pr = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
    pr = np.ascontiguousarray(pr)
    out = np.zeros((pr.shape[0], inp.D), dtype=np.float64)
    rc = _load().oracle_decode_fp8_pairs(
        _ptr(inp.q), _ptr(inp.k8), _ptr(inp.v8), _ptr(inp.ks), _ptr(inp.vs), _ptr(inp.bt),
        _ptr(inp.lens), inp.num_seqs, inp.H_q, inp.H_kv, inp.D, inp.maxb, inp.BS,
        inp.num_blocks, inp.scale, _ptr(pr), pr.shape[0], _ptr(out), int(num_threads))
    if rc != 0:
        raise OracleError(f"oracle rejected the input: {ERRORS.get(rc, rc)}")
    return out if pairs is not None else out.reshape(inp.num_seqs, inp.H_q, inp.D)


class XpackedInputs:
    """Host views of one decode problem over x-packed K [NB, H_kv, D/8, BS, 8]
    and D-major V [NB, H_kv, D, BS] (bf16)."""

    def __init__(self, q, kx, vt, block_tables, seq_lens, scale: float):
        self.q = _bits(q)
        self.kx = _bits(kx)
        self.vt = _bits(vt)
        self.bt = _i32(block_tables)
        self.lens = _i32(seq_lens)
        if self.q.ndim != 3 or self.kx.ndim != 5 or self.vt.ndim != 4:
            raise ValueError("q must be [S,H_q,D], K [NB,H_kv,D/8,BS,8] and V [NB,H_kv,D,BS]")
        self.num_seqs, self.H_q, self.D = self.q.shape
        self.num_blocks, self.H_kv, dx, self.BS, x = self.kx.shape
        if x != 8 or dx * 8 != self.D or self.vt.shape != (self.num_blocks, self.H_kv, self.D,
                                                              self.BS):
            raise ValueError("cache shapes do not match q's head_dim")
        self.maxb = self.bt.shape[1]
        self.scale = float(np.float32(scale))

    @classmethod
    def from_workload(cls, w) -> "XpackedInputs":
        return cls(w.q, w.kx, w.vt, w.block_tables, w.seq_lens, w.scale)


def decode_xpacked(x, pairs: Optional[Sequence[Sequence[int]]] = None,
                   num_threads: int = 0) -> np.ndarray:
    """The definition in float64 over x-packed K and D-major V; see the C source."""
    inp = x if isinstance(x, XpackedInputs) else XpackedInputs.from_workload(x)
    if pairs is None:
        pr = np.stack(np.meshgrid(np.arange(inp.num_seqs), np.arange(inp.H_q), indexing="ij"),
                      axis=-1).reshape(-1, 2).astype(np.int32)
    else:
        pr = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
    pr = np.ascontiguousarray(pr)
    out = np.zeros((pr.shape[0], inp.D), dtype=np.float64)
    rc = _load().oracle_decode_xpacked_pairs(
        _ptr(inp.q), _ptr(inp.kx), _ptr(inp.vt), _ptr(inp.bt), _ptr(inp.lens), inp.num_seqs,
        inp.H_q, inp.H_kv, inp.D, inp.maxb, inp.BS, inp.num_blocks, inp.scale, _ptr(pr),
        pr.shape[0], _ptr(out), int(num_threads))
    if rc != 0:
        raise OracleError(f"oracle rejected the input: {ERRORS.get(rc, rc)}")
    return out if pairs is not None else out.reshape(inp.num_seqs, inp.H_q, inp.D)


def decode_multi(x: Inputs, qo_indptr, causal: bool = True, num_threads: int = 0) -> np.ndarray:
    """Multi-token decode in float64 (see the C source): ``x.q`` holds the
    [total_q, H_q, D] query rows, sequence s owning rows qo_indptr[s] ..
    qo_indptr[s+1] - 1 (its last tokens); returns [total_q, H_q, D]."""
    qo = _i32(qo_indptr)
    if qo.shape != (len(x.lens) + 1,) or int(qo[-1]) != x.q.shape[0]:
        raise ValueError("qo_indptr must be [num_seqs + 1] ending at q's row count")
    out = np.zeros(x.q.shape, dtype=np.float64)
    rc = _load().oracle_decode_multi(
        _ptr(x.q), _ptr(x.k), _ptr(x.v), _ptr(qo), _ptr(x.bt), _ptr(x.lens), len(x.lens),
        x.H_q, x.H_kv, x.D, x.maxb, x.BS, x.num_blocks, x.scale, int(bool(causal)), _ptr(out),
        int(num_threads))
    if rc != 0:
        raise OracleError(f"oracle rejected the input: {ERRORS.get(rc, rc)}")
    return out


class MultiInputs(Inputs):
    """Inputs whose q holds any number of query rows ([total_q, H_q, D]); the
    sequence count comes from seq_lens."""

    def __init__(self, q, k_cache, v_cache, block_tables, seq_lens, scale: float):
        self.q = _bits(q)
        self.k = _bits(k_cache)
        self.v = _bits(v_cache)
        self.bt = _i32(block_tables)
        self.lens = _i32(seq_lens)
        if self.q.ndim != 3 or self.k.ndim != 4 or self.k.shape != self.v.shape:
            raise ValueError("q must be [total_q,H_q,D] and the caches [NB,H_kv,BS,D]")
        _, self.H_q, self.D = self.q.shape
        self.num_seqs = len(self.lens)
        self.num_blocks, self.H_kv, self.BS, Dk = self.k.shape
        if Dk != self.D or self.bt.shape[0] != self.num_seqs:
            raise ValueError("shapes disagree")
        self.maxb = self.bt.shape[1]
        self.scale = float(np.float32(scale))


def e4m3_table() -> np.ndarray:
    """The oracle's e4m3 decoding of the 256 byte codes."""
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def pieces(x, pairs, ranges):
    """Softmax pieces (M, l, o) of rows (s, h) over token ranges [t0, t1)."""
    inp = _as_inputs(x)
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    rg = np.ascontiguousarray(np.asarray(ranges, dtype=np.int32).reshape(-1, 2))
    if pr.shape != rg.shape:
        raise ValueError("one range per pair")
    n = pr.shape[0]
    M = np.zeros(n, dtype=np.float64)
    l = np.zeros(n, dtype=np.float64)
    o = np.zeros((n, inp.D), dtype=np.float64)
    rc = _load().oracle_partial_pairs(*inp._common(), _ptr(pr), _ptr(rg), n, _ptr(M), _ptr(l),
                                      _ptr(o))
    if rc != 0:
        raise OracleError(f"oracle rejected the input: {ERRORS.get(rc, rc)}")
    return M, l, o


def combine(a, b):
    """Merge two partial states (M, l, o): the binary op of the split-KV design.

    new_M = max(M_a, M_b); each side is weighted by exp(M_side - new_M); a side
    whose M is -inf (an empty range) gets weight zero.
    """
    Ma, la, oa = a
    Mb, lb, ob = b
    M = max(Ma, Mb)
    if M == -np.inf:
        return (M, 0.0, np.zeros_like(oa))
    wa = 0.0 if Ma == -np.inf else float(np.exp(Ma - M))
    wb = 0.0 if Mb == -np.inf else float(np.exp(Mb - M))
    return (M, wa * la + wb * lb, wa * oa + wb * ob)


def append(x, k_new, v_new) -> Inputs:
    """Cache append ("reshape and cache") of one new token per sequence.

    The paged-decode layout of the "Add Cuda Kernel" tutorial
    (include/kernels/attention.cuh, "Paged Attention - Decode") counts the new
    token in seq_lens, so its K and V must already sit in the cache when the
    decode runs; AstrAI's CUDA-kernels page (Backend Layer) has the backend own
    that write.  The new token of sequence s is position t = L_s - 1, and for
    every KV head g

        k_cache[bt[s, t // BS], g, t % BS, :] = k_new[s, g, :]   (v likewise).

    A sequence with L_s = 0 has no token and writes nothing.  ``k_new`` and
    ``v_new`` are [num_seqs, H_kv, D] bf16.  Returns new Inputs whose caches
    are copies with those rows written (the input is not modified).
    """
    inp = _as_inputs(x)
    kn = _bits(k_new)
    vn = _bits(v_new)
    if kn.shape != (inp.num_seqs, inp.H_kv, inp.D) or vn.shape != kn.shape:
        raise ValueError("k_new and v_new must be [num_seqs, H_kv, D]")
    out = copy.copy(inp)
    out.k = inp.k.copy()
    out.v = inp.v.copy()
    for s in range(inp.num_seqs):
        L = int(inp.lens[s])
        if L <= 0:
            continue
        if L > inp.maxb * inp.BS:
            raise OracleError(f"oracle rejected the input: {ERRORS[-3]}")
        t = L - 1
        b = int(inp.bt[s, t // inp.BS])
        if not 0 <= b < inp.num_blocks:
            raise OracleError(f"oracle rejected the input: {ERRORS[-4]}")
        out.k[b, :, t % inp.BS, :] = kn[s]
        out.v[b, :, t % inp.BS, :] = vn[s]
    return out


def finish(state) -> np.ndarray:
    """Normalise a merged state: o / l (zeros for an empty state)."""
    M, l, o = state
    if l == 0.0:
        return np.zeros_like(o)
    return o / l


def e4m3_encode(x) -> np.ndarray:
    """e4m3 codes of float32 values: the nearest e4m3 value, ties to the even
    code, magnitudes beyond 448 saturating to 448's code, NaN to 0x7F."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32).reshape(-1))
    out = np.zeros(a.shape[0], dtype=np.uint8)
    _load().oracle_e4m3_encode(_ptr(a), a.shape[0], _ptr(out))
    return out.reshape(np.shape(x))


def quantize_rows_e4m3(rows):
    """FP8 quantization of bf16 rows (last axis = one row): returns (codes uint8
    of the same shape, float32 dequant factor per row).  The factor is
    max|x| / 448 in float32 (1 for an all-zero row) and code = e4m3(x / factor)
    with a float32 quotient; see the C source for the reading of the pages."""
    b = _bits(rows)
    D = b.shape[-1]
    flat = np.ascontiguousarray(b.reshape(-1, D))
    codes = np.zeros(flat.shape, dtype=np.uint8)
    f = np.zeros(flat.shape[0], dtype=np.float32)
    _load().oracle_quantize_rows_e4m3(_ptr(flat), flat.shape[0], D, _ptr(codes), _ptr(f))
    return codes.reshape(b.shape), f.reshape(b.shape[:-1])


def append_fp8(x, k_new, v_new) -> "Fp8Inputs":
    """Cache append into FP8 caches: the write of ``append`` (the new token of
    sequence s is position L_s - 1), each new K and V row of every KV head
    quantized by ``quantize_rows_e4m3`` into its e4m3 bytes and its row float.
    ``k_new`` / ``v_new`` are [num_seqs, H_kv, D] bf16.  Returns new Fp8Inputs
    with those rows written (the input is not modified)."""
    inp = x if isinstance(x, Fp8Inputs) else Fp8Inputs.from_workload(x)
    kn = _bits(k_new)
    vn = _bits(v_new)
    if kn.shape != (inp.num_seqs, inp.H_kv, inp.D) or vn.shape != kn.shape:
        raise ValueError("k_new and v_new must be [num_seqs, H_kv, D]")
    kc, kf = quantize_rows_e4m3(kn)
    vc, vf = quantize_rows_e4m3(vn)
    out = copy.copy(inp)
    out.k8, out.v8 = inp.k8.copy(), inp.v8.copy()
    out.ks, out.vs = inp.ks.copy(), inp.vs.copy()
    for s in range(inp.num_seqs):
        L = int(inp.lens[s])
        if L <= 0:
            continue
        if L > inp.maxb * inp.BS:
            raise OracleError(f"oracle rejected the input: {ERRORS[-3]}")
        t = L - 1
        b = int(inp.bt[s, t // inp.BS])
        if not 0 <= b < inp.num_blocks:
            raise OracleError(f"oracle rejected the input: {ERRORS[-4]}")
        out.k8[b, :, t % inp.BS, :] = kc[s]
        out.v8[b, :, t % inp.BS, :] = vc[s]
        out.ks[b, :, t % inp.BS] = kf[s]
        out.vs[b, :, t % inp.BS] = vf[s]
    return out


def append_multi(x, qo_indptr, k_new, v_new) -> Inputs:
    """Cache append of several new tokens per sequence (the multi-token decode's
    write; rows located through qo_indptr as on AstrAI's CUDA Kernels page, "Q
    Scheduling and KV Addressing").  Sequence s owns rows qo_indptr[s] ..
    qo_indptr[s+1] - 1 of ``k_new`` / ``v_new`` ([total_q, H_kv, D] bf16): its
    last q_len tokens, row qo_indptr[s] + i being token t = L_s - q_len + i, so

        k_cache[bt[s, t // BS], g, t % BS, :] = k_new[qo_indptr[s] + i, g, :]

    for every KV head g (v alike).  Rows with t < 0 (more new rows than the
    sequence holds) write nothing.  Returns new Inputs with those rows written."""
    inp = _as_inputs(x)
    qo = _i32(qo_indptr)
    kn = _bits(k_new)
    vn = _bits(v_new)
    if qo.shape != (inp.num_seqs + 1,) or qo[0] != 0 or np.any(np.diff(qo) < 0):
        raise ValueError("qo_indptr must be [num_seqs + 1], non-decreasing from 0")
    total_q = int(qo[-1])
    if kn.shape != (total_q, inp.H_kv, inp.D) or vn.shape != kn.shape:
        raise ValueError("k_new and v_new must be [total_q, H_kv, D]")
    out = copy.copy(inp)
    out.k = inp.k.copy()
    out.v = inp.v.copy()
    for s in range(inp.num_seqs):
        L = int(inp.lens[s])
        if L > inp.maxb * inp.BS:
            raise OracleError(f"oracle rejected the input: {ERRORS[-3]}")
        ql = int(qo[s + 1] - qo[s])
        for i in range(ql):
            t = L - ql + i
            if t < 0:
                continue
            b = int(inp.bt[s, t // inp.BS])
            if not 0 <= b < inp.num_blocks:
                raise OracleError(f"oracle rejected the input: {ERRORS[-4]}")
            r = int(qo[s]) + i
            out.k[b, :, t % inp.BS, :] = kn[r]
            out.v[b, :, t % inp.BS, :] = vn[r]
    return out
