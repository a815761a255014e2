"""Seeded synthetic inputs for single-token paged-KV GQA decode attention.

This module draws random numbers and lays out the physical block pool; it
holds none of the attention arithmetic.  The FP64 oracle (``oracle/``) and the
CUDA path (``paged_kv_gqa_decode_gb300``) both consume what it makes, and
neither imports the other.

Layout (the paged-decode header of the "Add Cuda Kernel" tutorial, RL.cu
``include/kernels/attention.cuh``, "Paged Attention - Decode"):

* ``q``            ``[num_seqs, H_q, D]``                      bf16
* ``k_cache``      ``[num_blocks, H_kv, block_size, D]``       bf16
* ``v_cache``      ``[num_blocks, H_kv, block_size, D]``       bf16
* ``block_tables`` ``[num_seqs, max_blocks_per_seq]``          int32
* ``seq_lens``     ``[num_seqs]``                              int32

Recipe (the same for every workload):

* ``seq_lens`` come from ``numpy.random.default_rng(seed)`` (PCG64).
* The pool has ``sum_s ceil(L_s / block_size)`` data blocks plus spare
  blocks (one spare unless the workload fixes ``num_blocks``).  A seeded
  permutation of all physical block ids is dealt to the sequences in order;
  the first spare block of the permutation is the *poison* block, and every
  block-table entry a sequence does not use points at it.
* ``q``, ``K`` and ``V`` are drawn with a seeded ``torch.Generator`` on the
  target device (float32 normal, times the workload's standard deviation,
  rounded to bf16), in fixed-size chunks so the stream of draws does not
  depend on memory limits.
* ``poison`` fills every cache row that the definition never reads -- slots
  at or past ``L_s`` in a sequence's last page, every spare block -- with
  NaN (parity runs) or zero (timing runs).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np
import torch

__all__ = [
    "Spec",
    "Workload",
    "SPECS",
    "spec",
    "make",
    "custom_spec",
    "host_copy",
    "to_fp8",
    "Fp8Workload",
]


def _uniform_int(lo: int, hi: int) -> Callable[[np.random.Generator, int], np.ndarray]:
    def draw(rng: np.random.Generator, n: int) -> np.ndarray:
        return rng.integers(lo, hi, size=n, endpoint=True)

    return draw


def _log_uniform_int(lo: int, hi: int) -> Callable[[np.random.Generator, int], np.ndarray]:
    def draw(rng: np.random.Generator, n: int) -> np.ndarray:
        x = np.round(np.exp(rng.uniform(math.log(lo), math.log(hi), size=n)))
        return np.clip(x, lo, hi).astype(np.int64)

    return draw


def _fixed(values: Sequence[int]) -> Callable[[np.random.Generator, int], np.ndarray]:
    vals = np.asarray(values, dtype=np.int64)

    def draw(rng: np.random.Generator, n: int) -> np.ndarray:
        if n == len(vals):
            return vals.copy()
        return np.resize(vals, n)

    return draw


@dataclass(frozen=True)
class Spec:
    """Shape and value recipe of one synthetic decode workload."""

    name: str
    num_seqs: int
    H_q: int
    H_kv: int
    D: int
    block_size: int
    lens: Callable[[np.random.Generator, int], np.ndarray] = field(compare=False)
    max_len: int                     # upper bound of the length distribution
    q_std: float = 1.0
    kv_std: float = 1.0
    num_blocks: Optional[int] = None  # fixed pool size (else data blocks + 1)
    peaked_k_frac: float = 0.0        # fraction of K rows scaled by peaked_k_gain
    peaked_k_gain: float = 8.0
    scale: Optional[float] = None     # default 1/sqrt(D)
    description: str = ""

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, -(-self.max_len // self.block_size))

    @property
    def softmax_scale(self) -> float:
        return float(self.scale) if self.scale is not None else 1.0 / math.sqrt(self.D)


SPECS = {
    "tiny": Spec(
        "tiny", num_seqs=2, H_q=4, H_kv=2, D=64, block_size=16,
        lens=_fixed([37, 100]), max_len=100, num_blocks=16,
        description="tiny paged GQA decode: 2 seqs, H_q 4, H_kv 2, D 64, block 16, "
                    "seq_lens {37,100}, 16 shuffled blocks, scale 1/8"),
    "llama8b": Spec(
        "llama8b", num_seqs=32, H_q=32, H_kv=8, D=128, block_size=16,
        lens=_uniform_int(512, 4096), max_len=4096,
        description="LLaMA-3-8B-shaped decode: 32 seqs, H_q 32, H_kv 8, D 128, block 16, "
                    "seq_lens U[512,4096], shuffled blocks"),
    "qwen100k": Spec(
        "qwen100k", num_seqs=4, H_q=24, H_kv=4, D=256, block_size=16,
        lens=_fixed([100000] * 4), max_len=100000,
        description="Qwen-shaped long-context decode: 4 seqs x 100000 tokens, H_q 24, "
                    "H_kv 4, D 256, block 16, shuffled blocks"),
    "ragged256": Spec(
        "ragged256", num_seqs=256, H_q=32, H_kv=8, D=128, block_size=16,
        lens=_log_uniform_int(16, 32768), max_len=32768, peaked_k_frac=0.01,
        description="ragged large batch: 256 seqs, H_q 32, H_kv 8, D 128, block 16, "
                    "seq_lens log-uniform [16,32768], 1% of K rows x8"),
    "gqa8": Spec(
        "gqa8", num_seqs=64, H_q=64, H_kv=8, D=128, block_size=32,
        lens=_fixed([8192] * 64), max_len=8192, kv_std=0.5,
        description="GQA-8, bigger pages: 64 seqs x 8192 tokens, H_q 64, H_kv 8, D 128, "
                    "block 32, K/V std 0.5"),
}

# Seeds follow the workload's position in the published list (1000 + index).
SEEDS = {"tiny": 1000, "llama8b": 1001, "qwen100k": 1002, "ragged256": 1003, "gqa8": 1004}


def spec(name: str) -> Spec:
    return SPECS[name]


def custom_spec(name: str, num_seqs: int, H_q: int, H_kv: int, D: int, block_size: int,
                lens: Sequence[int], max_len: Optional[int] = None, **kw) -> Spec:
    """A workload with explicit sequence lengths (used by the edge-case tests)."""
    lens = [int(x) for x in lens]
    if max_len is None:
        max_len = max([1] + lens)
    return Spec(name, num_seqs=num_seqs, H_q=H_q, H_kv=H_kv, D=D, block_size=block_size,
                lens=_fixed(lens if lens else [0]), max_len=max_len, **kw)


@dataclass
class Workload:
    spec: Spec
    seed: int
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    num_blocks: int
    poison_block: int
    poison: str

    @property
    def scale(self) -> float:
        return self.spec.softmax_scale

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def lens_list(self):
        return [int(x) for x in self.seq_lens.cpu().tolist()]


_CHUNK_ELEMS = 1 << 26  # draws are made in chunks of this many elements


def _fill_normal(out: torch.Tensor, gen: torch.Generator, std: float) -> None:
    flat = out.view(-1)
    n = flat.numel()
    for i in range(0, n, _CHUNK_ELEMS):
        m = min(_CHUNK_ELEMS, n - i)
        x = torch.randn(m, generator=gen, device=out.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[i:i + m].copy_(x.to(torch.bfloat16))


def _scale_random_rows(k: torch.Tensor, gen: torch.Generator, frac: float, gain: float) -> None:
    """Multiply a Bernoulli(frac) subset of K rows (token, kv-head) by gain."""
    rows = k.view(-1, k.shape[-1])
    n = rows.shape[0]
    step = max(1, _CHUNK_ELEMS // max(1, k.shape[-1]))
    for i in range(0, n, step):
        m = min(step, n - i)
        u = torch.rand(m, generator=gen, device=k.device, dtype=torch.float32)
        sel = (u < frac).nonzero().view(-1) + i
        if sel.numel():
            rows[sel] = (rows[sel].float() * gain).to(torch.bfloat16)


def make(spec_or_name, seed: Optional[int] = None, device="cpu", poison: str = "nan",
         lens_override: Optional[Sequence[int]] = None) -> Workload:
    """Build one seeded workload on ``device``.

    ``poison`` is ``"nan"`` (parity: unread rows hold NaN), ``"zero"`` (timing)
    or ``"none"`` (leave the random values in place).
    """
    sp = SPECS[spec_or_name] if isinstance(spec_or_name, str) else spec_or_name
    if seed is None:
        seed = SEEDS.get(sp.name, 1234)
    rng = np.random.default_rng(seed)
    if lens_override is not None:
        lens = np.asarray(list(lens_override), dtype=np.int64)
    else:
        lens = np.asarray(sp.lens(rng, sp.num_seqs), dtype=np.int64)[: sp.num_seqs]
    if len(lens) != sp.num_seqs:
        raise ValueError("need one length per sequence")
    BS = sp.block_size
    maxb = sp.max_blocks_per_seq
    pages = [-(-int(L) // BS) if L > 0 else 0 for L in lens]
    if any(p > maxb for p in pages):
        raise ValueError("a sequence needs more pages than max_blocks_per_seq")
    needed = int(sum(pages))
    num_blocks = sp.num_blocks if sp.num_blocks is not None else needed + 1
    if num_blocks < needed + 1:
        raise ValueError("block pool too small for the sequences plus one poison block")

    perm = rng.permutation(num_blocks)
    poison_block = int(perm[needed])
    bt = np.full((sp.num_seqs, maxb), poison_block, dtype=np.int32)
    pos = 0
    for s, p in enumerate(pages):
        bt[s, :p] = perm[pos:pos + p]
        pos += p

    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    q = torch.empty((sp.num_seqs, sp.H_q, sp.D), dtype=torch.bfloat16, device=dev)
    k = torch.empty((num_blocks, sp.H_kv, BS, sp.D), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    _fill_normal(q, gen, sp.q_std)
    _fill_normal(k, gen, sp.kv_std)
    _fill_normal(v, gen, sp.kv_std)
    if sp.peaked_k_frac > 0:
        _scale_random_rows(k, gen, sp.peaked_k_frac, sp.peaked_k_gain)

    if poison in ("nan", "zero"):
        val = float("nan") if poison == "nan" else 0.0
        used = np.zeros(num_blocks, dtype=bool)
        used[perm[:needed]] = True
        spare = torch.from_numpy(np.nonzero(~used)[0]).to(dev)
        if spare.numel():
            k[spare] = val
            v[spare] = val
        for s, L in enumerate(lens):
            L = int(L)
            if L > 0 and L % BS:
                blk = int(bt[s, pages[s] - 1])
                k[blk, :, L % BS:, :] = val
                v[blk, :, L % BS:, :] = val
    elif poison != "none":
        raise ValueError(f"unknown poison mode {poison!r}")

    return Workload(
        spec=sp, seed=int(seed), q=q, k_cache=k, v_cache=v,
        block_tables=torch.from_numpy(bt).to(dev),
        seq_lens=torch.from_numpy(lens.astype(np.int32)).to(dev),
        num_blocks=num_blocks, poison_block=poison_block, poison=poison)


E4M3_MAX = 448.0  # largest finite e4m3 value


@dataclass
class Fp8Workload:
    """A workload whose caches are FP8: e4m3 bytes in the bf16 layout and one
    dequant float per (block, KV head, slot) for K and for V, so that
    element = e4m3 value x row float.  q, tables and lengths are the base's."""

    base: Workload
    k8: torch.Tensor       # uint8 [num_blocks, H_kv, BS, D]
    v8: torch.Tensor
    k_scale: torch.Tensor  # float32 [num_blocks, H_kv, BS]
    v_scale: torch.Tensor

    def __getattr__(self, name):  # q, block_tables, seq_lens, scale, spec, lens_list, ...
        return getattr(self.base, name)


def _quantize_rows(x: torch.Tensor):
    """Per-row (last axis) e4m3 quantization of a bf16 cache, chunked over blocks:
    the row float is max|x| / 448 (1 for an all-zero row; NaN rows stay NaN)."""
    q8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    step = max(1, (1 << 24) // max(1, x[0].numel()))
    for b0 in range(0, x.shape[0], step):
        xf = x[b0:b0 + step].float()
        amax = xf.abs().amax(dim=-1)
        s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        s = torch.where(torch.isnan(amax), amax, s)
        q8[b0:b0 + step] = (xf / s.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
        sc[b0:b0 + step] = s
    return q8, sc


def to_fp8(w: Workload) -> Fp8Workload:
    """The same problem with FP8 caches (the bf16 caches quantized per row)."""
    k8, ks = _quantize_rows(w.k_cache)
    v8, vs = _quantize_rows(w.v_cache)
    return Fp8Workload(base=w, k8=k8, v8=v8, k_scale=ks, v_scale=vs)


@dataclass
class XpackedWorkload:
    """A workload whose bf16 caches are in the x-packed K / D-major V layout:
    kx[b, g, d // 8, t, d % 8] = k_cache[b, g, t, d], vt[b, g, d, t] = v_cache[b, g, t, d]."""

    base: Workload
    kx: torch.Tensor  # bf16 [num_blocks, H_kv, D / 8, BS, 8]
    vt: torch.Tensor  # bf16 [num_blocks, H_kv, D, BS]

    def __getattr__(self, name):
        return getattr(self.base, name)


def to_xpacked(w: Workload) -> XpackedWorkload:
    """The same problem with its caches repacked (same values, other order)."""
    nb, hk, bs, d = w.k_cache.shape
    kx = w.k_cache.view(nb, hk, bs, d // 8, 8).permute(0, 1, 3, 2, 4).contiguous()
    vt = w.v_cache.permute(0, 1, 3, 2).contiguous()
    return XpackedWorkload(base=w, kx=kx, vt=vt)


def host_copy(w: Workload) -> Workload:
    """The same workload with every tensor copied to host memory."""
    return Workload(spec=w.spec, seed=w.seed, q=w.q.cpu(), k_cache=w.k_cache.cpu(),
                    v_cache=w.v_cache.cpu(), block_tables=w.block_tables.cpu(),
                    seq_lens=w.seq_lens.cpu(), num_blocks=w.num_blocks,
                    poison_block=w.poison_block, poison=w.poison)
