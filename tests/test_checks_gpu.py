"""Device-side input checks on every entry point (paged_attn_set_checks): a block id
outside the caller's pool is reported in the status word and never read, for the
bf16, FP8, x-packed and multi-token decodes and for every append; the rows of
the other sequences still match the oracle.  And the status word is written only
after the work ahead in the stream: under the early prologue a kernel that
zero-fills it just before the call cannot erase the report.

The layouts are those of the RL.cu "Add Cuda Kernel" tutorial (standard),
"Paged Attention Kernel Architecture for BI-V100" section 3 (x-packed), the
nvfp4-megamoe README "Stage D: FP8 Paged KV Gather" (FP8) and AstrAI's CUDA
Kernels page "Q Scheduling and KV Addressing" (multi-token rows)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import paged_kv_gqa_decode_gb300 as pa

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
BAD_BLOCK, BAD_LENGTH = 1, 2

LENS = [300, 17, 16, 1, 513, 64, 200, 33, 128, 999, 5, 250]
SPEC = workloads.custom_spec("checks", 12, 32, 8, 128, 16, LENS, max_len=1024)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_decode_gb300 import build

    build.build()
    pa.load()


@pytest.fixture
def status():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    yield st
    pa.paged_attn_set_checks(0, None)
    pa.paged_attn_set_launch_flags(0)


def bad_table(w):
    """The block table with one used entry of sequence 0 pointing one past the pool."""
    bt = w.block_tables.clone()
    bt[0, 3] = w.k_cache.shape[0]
    return bt


def others(out, ref):
    """Rows of every sequence but the first (whose page 3 is bad)."""
    got = out.float().cpu().double().numpy()[1:]
    assert np.isfinite(out.float().cpu().numpy()).all()
    err = np.abs(got - ref[1:])
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def test_decode_reports_a_bad_block_and_stays_in_the_pool(status):
    w = workloads.make(SPEC, seed=51, device="cuda", poison="nan")
    ref = oracle.decode(workloads.host_copy(w))
    pa.paged_attn_set_checks(w.k_cache.shape[0], status)
    out = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, bad_table(w), w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert int(status.item()) & BAD_BLOCK
    others(out, ref)
    # checks off: a good call writes nothing into the old status word
    pa.paged_attn_set_checks(0, None)
    status.zero_()
    pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_fp8_decode_reports_a_bad_block(status):
    w = workloads.make(SPEC, seed=52, device="cuda", poison="nan")
    f = workloads.to_fp8(w)
    host = oracle.Fp8Inputs(f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(), f.v_scale.cpu(),
                            f.block_tables.cpu(), f.seq_lens.cpu(), f.scale)
    ref = oracle.decode_fp8(host)
    pa.paged_attn_set_checks(f.k8.shape[0], status)
    out = pa.paged_attn_decode_fp8(f.q, f.k8, f.v8, f.k_scale, f.v_scale, bad_table(w),
                                   f.seq_lens, f.scale)
    torch.cuda.synchronize()
    assert int(status.item()) & BAD_BLOCK
    others(out, ref)


@pytest.mark.parametrize("bs", [16, 32])
def test_xpacked_decode_reports_a_bad_block(status, bs):
    sp = workloads.custom_spec("checks_xp", 12, 32, 8, 128, bs, LENS, max_len=1024)
    w = workloads.make(sp, seed=53, device="cuda", poison="nan")
    x = workloads.to_xpacked(w)
    ref = oracle.decode(workloads.host_copy(w))
    pa.paged_attn_set_checks(w.k_cache.shape[0], status)
    out = pa.paged_attn_decode_xpacked(w.q, x.kx, x.vt, bad_table(w), w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert int(status.item()) & BAD_BLOCK
    others(out, ref)


def test_multi_decode_reports_a_bad_block(status):
    w = workloads.make(SPEC, seed=54, device="cuda", poison="nan")
    qlens = [min(3, L) for L in w.lens_list]
    g = torch.Generator().manual_seed(55)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    q = torch.randn(int(qo[-1]), 32, 128, generator=g).to(torch.bfloat16)
    x = oracle.MultiInputs(q, w.k_cache.cpu(), w.v_cache.cpu(), w.block_tables.cpu(),
                           w.seq_lens.cpu(), w.scale)
    ref = oracle.decode_multi(x, qo)
    pa.paged_attn_set_checks(w.k_cache.shape[0], status)
    out = pa.paged_attn_decode_multi(q.cuda(), w.k_cache, w.v_cache, qo.cuda(), bad_table(w),
                                     w.seq_lens, w.scale, 3)
    torch.cuda.synchronize()
    assert int(status.item()) & BAD_BLOCK
    rows = int(qo[1])  # sequence 0's rows
    got = out.float().cpu().double().numpy()[rows:]
    err = np.abs(got - ref[rows:])
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS


def _rows(w, n, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (n, w.spec.H_kv, w.spec.D)
    return (torch.randn(shape, generator=g).to(torch.bfloat16).cuda(),
            torch.randn(shape, generator=g).to(torch.bfloat16).cuda())


def test_appends_skip_a_bad_block_and_report_it(status):
    """A sequence whose new token's block id is outside the pool: every append
    entry point writes nothing for it, reports bit 0, and writes the others."""
    lens = [40, 17, 33, 64]
    sp = workloads.custom_spec("checks_app", 4, 32, 8, 128, 16, lens, max_len=128)
    for kind in ("bf16", "decode", "multi", "fp8", "fp8_decode"):
        w = workloads.make(sp, seed=56, device="cuda", poison="nan")
        bt = w.block_tables.clone()
        bt[0, (lens[0] - 1) // 16] = w.k_cache.shape[0]  # the new token's page of sequence 0
        k_new, v_new = _rows(w, 4, 57)
        status.zero_()
        pa.paged_attn_set_checks(w.k_cache.shape[0], status)
        if kind in ("bf16", "decode", "multi"):
            before = w.k_cache.clone()
            if kind == "bf16":
                pa.paged_kv_append(k_new, v_new, w.k_cache, w.v_cache, bt, w.seq_lens)
            elif kind == "decode":
                pa.paged_attn_append_decode(w.q, k_new, v_new, w.k_cache, w.v_cache, bt,
                                            w.seq_lens, w.scale)
            else:
                qo = torch.arange(5, dtype=torch.int32, device="cuda")
                pa.paged_kv_append_multi(k_new, v_new, w.k_cache, w.v_cache, qo, bt, w.seq_lens)
            torch.cuda.synchronize()
            changed = (w.k_cache.view(torch.int16) != before.view(torch.int16)).sum().item()
            assert changed <= 3 * 8 * 128, kind  # sequence 0's rows were not written
        else:
            f = workloads.to_fp8(w)
            b8 = f.k8.clone()
            if kind == "fp8":
                pa.paged_kv_append_fp8(k_new, v_new, f.k8, f.v8, f.k_scale, f.v_scale, bt,
                                       f.seq_lens)
            else:
                pa.paged_attn_append_decode_fp8(f.q, k_new, v_new, f.k8, f.v8, f.k_scale,
                                                f.v_scale, bt, f.seq_lens, f.scale)
            torch.cuda.synchronize()
            changed = (f.k8 != b8).sum().item()
            assert changed <= 3 * 8 * 128, kind
        assert int(status.item()) & BAD_BLOCK, kind
        pa.paged_attn_set_checks(0, None)


def test_status_is_written_after_the_work_ahead(status):
    """Under the early prologue the producer scans the lengths before the work ahead
    has finished; a bad length found there must still be reported after that work
    (here: a kernel zero-filling the status word just before the call)."""
    w = workloads.make(SPEC, seed=58, device="cuda", poison="nan")
    sl = w.seq_lens.clone()
    sl[2] = 10**6  # past max_blocks_per_seq * block_size
    pa.paged_attn_set_launch_flags(pa.FLAG_EARLY_PROLOGUE)
    for _ in range(5):
        status.fill_(7 << 8)  # a kernel writing the word...
        status.zero_()        # ...and zero-filling it right before the decode
        pa.paged_attn_decode_checked(w.q, w.k_cache, w.v_cache, w.block_tables, sl, w.scale,
                                     status)
        torch.cuda.synchronize()
        assert int(status.item()) == BAD_LENGTH


def test_set_checks_rejects_bad_arguments():
    lib = pa.load()
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert lib.paged_attn_set_checks(0, None) == 0
    assert lib.paged_attn_set_checks(-3, st.data_ptr()) == -5
    assert lib.paged_attn_set_checks(10, None) == -1
    assert lib.paged_attn_set_checks(10, st.data_ptr() + 2) == -1
    assert lib.paged_attn_set_checks(0, None) == 0
