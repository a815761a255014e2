"""The online softmax under score patterns that move its running maximum in
every way: scores rising page after page (by about one unit of log2 per page,
so the kernels' lazily raised maximum trails the true one and is raised every
few pages), falling, isolated spikes far above the rest, and an oscillation
about as wide as the lag the kernels allow.  Each decode entry point (bf16,
FP8, x-packed, multi-token causal) is held to the FP64 oracle at the parity
tolerance.

The definition is the RL.cu tutorial's "Paged Attention - Decode" (softmax of
scale * q . K_t over t < seq_len, then the weighted sum of V_t); the FP8 and
x-packed layouts are those of the nvfp4-megamoe README "Stage D: FP8 Paged KV
Gather" and "Paged Attention Kernel Architecture for BI-V100" section 3, the
multi-token rows AstrAI's CUDA Kernels page "Q Scheduling and KV Addressing".
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import paged_kv_gqa_decode_gb300 as pa

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
LENS = [700, 333, 1000, 64, 257]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_decode_gb300 import build

    build.build()
    pa.load()


def ramp(s, L):
    """Column 0 of K for the tokens of sequence s (q's column 0 is 1, so with
    the softmax scale 1/sqrt(128) a value of 450 is a score of ~40, ~57 in log2)."""
    t = torch.arange(L, dtype=torch.float64)
    if s % 5 == 0:
        return 450.0 * t / L  # rises through the whole sequence
    if s % 5 == 1:
        return 450.0 * (1.0 - t / L)  # falls
    if s % 5 == 2:
        r = torch.zeros(L, dtype=torch.float64)
        r[[5, L // 2, L - 1]] = 300.0  # spikes
        return r
    if s % 5 == 3:
        return 40.0 * torch.sin(t / 3.0)  # oscillates about as wide as the allowed lag
    return -450.0 * t / L + 60.0 * (t > L - 20)  # falls, then jumps near the end


def make(seed, BS=16, H_q=16, H_kv=2):
    sp = workloads.custom_spec("softmax_ramps", len(LENS), H_q, H_kv, 128, BS, LENS,
                               max_len=1024)
    w = workloads.make(sp, seed=seed, device="cuda", poison="nan")
    bt = w.block_tables.cpu()
    for s, L in enumerate(w.lens_list):
        t = torch.arange(L)
        blocks = bt[s, t // BS].long().cuda()
        slots = (t % BS).cuda()
        w.k_cache[blocks, :, slots, 0] = ramp(s, L).to(torch.bfloat16).cuda()[:, None]
    w.q[:, :, 0] = 1.0
    return w


def check(out, ref, what):
    got = out.float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (what, err.max(), err.mean())


@pytest.mark.parametrize("BS", [16, 32])
def test_bf16_decode_follows_moving_maxima(BS):
    w = make(71 + BS, BS=BS)
    out = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    check(out, oracle.decode(workloads.host_copy(w)), f"bf16 BS {BS}")


def test_gqa16_decode_follows_moving_maxima():
    w = make(75, H_q=32, H_kv=2)  # G = 16: two n-tiles of heads
    out = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    check(out, oracle.decode(workloads.host_copy(w)), "G 16")


@pytest.mark.parametrize("BS", [16, 32])
def test_fp8_decode_follows_moving_maxima(BS):
    w = make(81 + BS, BS=BS)
    f = workloads.to_fp8(w)
    out = pa.paged_attn_decode_fp8(f.q, f.k8, f.v8, f.k_scale, f.v_scale, f.block_tables,
                                   f.seq_lens, f.scale)
    torch.cuda.synchronize()
    host = oracle.Fp8Inputs(f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(), f.v_scale.cpu(),
                            f.block_tables.cpu(), f.seq_lens.cpu(), f.scale)
    check(out, oracle.decode_fp8(host), f"FP8 BS {BS}")


def test_xpacked_decode_follows_moving_maxima():
    w = make(91)
    x = workloads.to_xpacked(w)
    out = pa.paged_attn_decode_xpacked(w.q, x.kx, x.vt, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    check(out, oracle.decode(workloads.host_copy(w)), "x-packed")


@pytest.mark.parametrize("q_len", [2, 5])
def test_multi_token_decode_follows_moving_maxima(q_len):
    w = make(95 + q_len)
    qo = torch.tensor(np.arange(len(LENS) + 1) * q_len, dtype=torch.int32)
    g = torch.Generator().manual_seed(97)
    q = torch.randn(int(qo[-1]), w.spec.H_q, 128, generator=g).to(torch.bfloat16)
    q[:, :, 0] = 1.0
    out = pa.paged_attn_decode_multi(q.cuda(), w.k_cache, w.v_cache, qo.cuda(), w.block_tables,
                                     w.seq_lens, w.scale, q_len)
    torch.cuda.synchronize()
    mi = oracle.MultiInputs(q, w.k_cache.cpu(), w.v_cache.cpu(), w.block_tables.cpu(),
                            w.seq_lens.cpu(), w.scale)
    check(out, oracle.decode_multi(mi, qo), f"multi q_len {q_len}")
