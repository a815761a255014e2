"""GPU parity of the decode over x-packed K / D-major V caches: against the
oracle's x-packed definition (float64) on the published workloads and a shape /
tail sweep, and bit for bit against the standard-layout decode of the same
values (the arithmetic is the same; only the shared-memory addressing differs)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import paged_kv_gqa_decode_gb300 as pa

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_decode_gb300 import build

    build.build()
    pa.load()


def run_xp(x):
    out = pa.paged_attn_decode_xpacked(x.q, x.kx, x.vt, x.block_tables, x.seq_lens, x.scale)
    torch.cuda.synchronize()
    return out


def reference(x):
    host = oracle.XpackedInputs(x.q.cpu(), x.kx.cpu(), x.vt.cpu(), x.block_tables.cpu(),
                                x.seq_lens.cpu(), x.scale)
    return oracle.decode_xpacked(host)


def assert_parity(out, ref, what=""):
    got = out.float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, \
        f"{what}: max {err.max():.3e} mean {err.mean():.3e}"


@pytest.mark.parametrize("name", ["tiny", "llama8b", "qwen100k", "ragged256", "gqa8"])
def test_published_workloads_xpacked(name):
    w = workloads.make(name, device="cuda", poison="nan")
    x = workloads.to_xpacked(w)
    out = run_xp(x)
    assert_parity(out, reference(x), name)
    std = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), std.view(torch.int16)), name


EDGE_LENS = [0, 1, 15, 16, 17, 31, 32, 33, 100, 257, 1000]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (8, 2), (12, 2), (16, 1)])
def test_xpacked_shapes_and_ragged_tails(D, BS, H_q, H_kv):
    sp = workloads.custom_spec("xpsweep", len(EDGE_LENS), H_q, H_kv, D, BS, EDGE_LENS,
                               max_len=1024)
    w = workloads.make(sp, seed=D + BS + H_q, device="cuda", poison="nan")
    x = workloads.to_xpacked(w)
    out = run_xp(x)
    assert_parity(out, reference(x), f"D{D} BS{BS} G{H_q // H_kv}")
    assert torch.count_nonzero(out[0]).item() == 0  # the empty sequence
    std = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), std.view(torch.int16))


def test_xpacked_long_sequence_split_over_all_ctas():
    sp = workloads.custom_spec("one", 1, 8, 1, 128, 16, [60000])
    x = workloads.to_xpacked(workloads.make(sp, seed=3, device="cuda"))
    assert_parity(run_xp(x), reference(x))


def test_xpacked_rejects_bad_arguments():
    w = workloads.make("tiny", device="cuda")
    x = workloads.to_xpacked(w)
    with pytest.raises(ValueError):
        pa.paged_attn_decode_xpacked(x.q, x.kx[..., :4].contiguous(), x.vt, x.block_tables,
                                     x.seq_lens, x.scale)
    lib = pa.load()
    assert lib.paged_attn_decode_xpacked(0, 0, 0, 0, 0, 0, 2, 4, 2, 64, 7, 16, 0.125, 0) == -1
    rc = lib.paged_attn_decode_xpacked(x.q.data_ptr(), x.kx.data_ptr(), x.vt.data_ptr(),
                                       x.q.data_ptr(), x.block_tables.data_ptr(),
                                       x.seq_lens.data_ptr(), 2, 4, 2, 96, 7, 16, 0.125, 0)
    assert rc == -3  # head_dim


def test_xpacked_more_sequences_than_one_launch_holds():
    lens = list(np.random.default_rng(15).integers(1, 70, size=5000))
    sp = workloads.custom_spec("wide", len(lens), 4, 1, 64, 32, lens, max_len=96)
    w = workloads.make(sp, seed=15, device="cuda", poison="nan")
    x = workloads.to_xpacked(w)
    assert_parity(run_xp(x), reference(x), "5000 sequences")
