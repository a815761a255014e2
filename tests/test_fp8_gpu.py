"""GPU parity of the decode over FP8 caches against the oracle's FP8 definition
(e4m3 values times their row's float, in float64), on the published workloads
quantized per cache row, a shape / tail sweep, and NaN-poisoned unread rows."""
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


def run_fp8(f):
    out = pa.paged_attn_decode_fp8(f.q, f.k8, f.v8, f.k_scale, f.v_scale, f.block_tables,
                                   f.seq_lens, f.scale)
    torch.cuda.synchronize()
    return out


def reference(f):
    host = oracle.Fp8Inputs(f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(), f.v_scale.cpu(),
                            f.block_tables.cpu(), f.seq_lens.cpu(), f.scale)
    return oracle.decode_fp8(host)


def assert_parity(out, ref, what=""):
    got = out.float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, \
        f"{what}: max {err.max():.3e} mean {err.mean():.3e}"


@pytest.mark.parametrize("name", ["llama8b", "qwen100k", "ragged256", "gqa8"])
def test_published_workloads_fp8(name):
    f = workloads.to_fp8(workloads.make(name, device="cuda", poison="nan"))
    assert_parity(run_fp8(f), reference(f), name)


EDGE_LENS = [0, 1, 15, 16, 17, 31, 32, 33, 100, 257, 1000]


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (8, 2), (12, 2), (24, 2), (16, 1)])
def test_fp8_shapes_and_ragged_tails(D, BS, H_q, H_kv):
    sp = workloads.custom_spec("fp8sweep", len(EDGE_LENS), H_q, H_kv, D, BS, EDGE_LENS,
                               max_len=1024)
    f = workloads.to_fp8(workloads.make(sp, seed=D + BS + H_q, device="cuda", poison="nan"))
    out = run_fp8(f)
    assert_parity(out, reference(f), f"D{D} BS{BS} G{H_q // H_kv}")
    assert torch.count_nonzero(out[0]).item() == 0  # the empty sequence


def test_fp8_long_sequence_split_over_all_ctas():
    sp = workloads.custom_spec("one", 1, 8, 1, 128, 16, [60000])
    f = workloads.to_fp8(workloads.make(sp, seed=3, device="cuda"))
    assert_parity(run_fp8(f), reference(f))


def test_fp8_repeat_calls_are_bitwise_identical():
    f = workloads.to_fp8(workloads.make("ragged256", device="cuda", poison="nan"))
    a = run_fp8(f).clone()
    b = run_fp8(f)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_fp8_stays_close_to_the_bf16_decode():
    """Quantization error of the cache, end to end (the pages report cosine 0.9997)."""
    w = workloads.make("llama8b", device="cuda", poison="zero")
    f = workloads.to_fp8(w)
    a = run_fp8(f).float().flatten()
    b = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.scale).float().flatten()
    cos = torch.dot(a, b) / (a.norm() * b.norm())
    assert cos.item() > 0.999


def test_fp8_rejects_head_dim_64():
    f = workloads.to_fp8(workloads.make("tiny", device="cuda"))
    with pytest.raises(pa.PagedAttnError) as e:
        run_fp8(f)
    assert e.value.status == -3


def test_fp8_more_sequences_than_one_launch_holds():
    lens = list(np.random.default_rng(14).integers(1, 70, size=5000))
    sp = workloads.custom_spec("wide", len(lens), 4, 1, 128, 16, lens, max_len=80)
    f = workloads.to_fp8(workloads.make(sp, seed=14, device="cuda", poison="nan"))
    assert_parity(run_fp8(f), reference(f), "5000 sequences")
