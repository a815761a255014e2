"""GPU parity of the cache append: the standalone kernel and the append fused
into the decode launch, against the oracle's append (and decode) on the same
seeded inputs.  The written cache rows are compared bit for bit; the decode
output within the decode's tolerance."""
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


def new_rows(w, seed):
    """Seeded bf16 rows for each sequence's new token, [num_seqs, H_kv, D] on the device."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (w.spec.num_seqs, w.spec.H_kv, w.spec.D)
    k = torch.randn(shape, generator=g).to(torch.bfloat16)
    v = torch.randn(shape, generator=g).to(torch.bfloat16)
    return k.cuda(), v.cuda()


def expected(w, k_new, v_new):
    return oracle.append(workloads.host_copy(w), k_new, v_new)


def cache_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_parity(out, ref, what=""):
    got = out.float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, \
        f"{what}: max {err.max():.3e} mean {err.mean():.3e}"


EDGE = workloads.custom_spec("append_edges", 10, 8, 2, 128, 16,
                             [1, 15, 16, 17, 31, 32, 33, 0, 48, 1000], max_len=1024)


@pytest.mark.parametrize("name", ["tiny", "edges", "llama8b", "ragged256"])
def test_standalone_append_writes_exactly_the_oracle_rows(name):
    w = workloads.make(EDGE if name == "edges" else name, seed=21, device="cuda", poison="nan")
    k_new, v_new = new_rows(w, 5)
    exp = expected(w, k_new, v_new)
    pa.paged_kv_append(k_new, v_new, w.k_cache, w.v_cache, w.block_tables, w.seq_lens)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(w.k_cache), exp.k)
    assert np.array_equal(cache_bits(w.v_cache), exp.v)


@pytest.mark.parametrize("name", ["tiny", "edges", "llama8b", "qwen100k", "ragged256", "gqa8"])
def test_fused_append_decode_matches_oracle(name):
    w = workloads.make(EDGE if name == "edges" else name, seed=22, device="cuda", poison="nan")
    k_new, v_new = new_rows(w, 6)
    exp = expected(w, k_new, v_new)
    out = pa.paged_attn_append_decode(w.q, k_new, v_new, w.k_cache, w.v_cache, w.block_tables,
                                      w.seq_lens, w.scale)
    torch.cuda.synchronize()
    # the rows landed in the caches, nothing else changed ...
    assert np.array_equal(cache_bits(w.k_cache), exp.k)
    assert np.array_equal(cache_bits(w.v_cache), exp.v)
    # ... and the decode saw them
    assert_parity(out, oracle.decode(exp), name)


@pytest.mark.parametrize("name", ["edges", "llama8b", "qwen100k"])
def test_fused_equals_append_then_decode(name):
    """The fused launch gives bit for bit what the two separate calls give."""
    sp = EDGE if name == "edges" else workloads.spec(name)
    w1 = workloads.make(sp, seed=23, device="cuda", poison="nan")
    w2 = workloads.make(sp, seed=23, device="cuda", poison="nan")
    k_new, v_new = new_rows(w1, 7)
    fused = pa.paged_attn_append_decode(w1.q, k_new, v_new, w1.k_cache, w1.v_cache,
                                        w1.block_tables, w1.seq_lens, w1.scale)
    pa.paged_kv_append(k_new, v_new, w2.k_cache, w2.v_cache, w2.block_tables, w2.seq_lens)
    plain = pa.paged_attn_decode(w2.q, w2.k_cache, w2.v_cache, w2.block_tables, w2.seq_lens,
                                 w2.scale)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), plain.view(torch.int16))
    assert torch.equal(w1.k_cache.view(torch.int16), w2.k_cache.view(torch.int16))


def test_one_token_sequences_decode_to_their_new_v():
    sp = workloads.custom_spec("ones", 40, 8, 2, 128, 16, [1] * 40)
    w = workloads.make(sp, seed=24, device="cuda", poison="nan")
    k_new, v_new = new_rows(w, 8)
    out = pa.paged_attn_append_decode(w.q, k_new, v_new, w.k_cache, w.v_cache, w.block_tables,
                                      w.seq_lens, w.scale)
    torch.cuda.synchronize()
    want = v_new.repeat_interleave(4, dim=1)  # G = 4 query heads per KV head
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("num_seqs,H_kv", [(1100, 1), (700, 8)])
def test_many_short_sequences(num_seqs, H_kv):
    # 1100 x 1 KV head: fused, nearly every page is the last of its piece;
    # 700 x 8: enough pieces per CTA that the call runs the append apart
    lens = list(np.random.default_rng(25).integers(0, 40, size=num_seqs))
    sp = workloads.custom_spec("short", len(lens), 8, H_kv, 64, 16, lens, max_len=48)
    w = workloads.make(sp, seed=25, device="cuda", poison="nan")
    k_new, v_new = new_rows(w, 9)
    exp = expected(w, k_new, v_new)
    out = pa.paged_attn_append_decode(w.q, k_new, v_new, w.k_cache, w.v_cache, w.block_tables,
                                      w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(w.k_cache), exp.k)
    assert_parity(out, oracle.decode(exp), "short")


def test_append_rejects_bad_arguments():
    w = workloads.make("tiny", device="cuda")
    k_new, v_new = new_rows(w, 1)
    with pytest.raises(ValueError):
        pa.paged_kv_append(k_new[:, :1], v_new, w.k_cache, w.v_cache, w.block_tables, w.seq_lens)
    lib = pa.load()
    rc = lib.paged_kv_append(0, 0, 0, 0, 0, 0, 2, 2, 64, 7, 16, 0)
    assert rc == -1  # null pointers
    rc = lib.paged_kv_append(k_new.data_ptr(), v_new.data_ptr(), w.k_cache.data_ptr(),
                             w.v_cache.data_ptr(), w.block_tables.data_ptr(),
                             w.seq_lens.data_ptr(), 2, 2, 96, 7, 16, 0)
    assert rc == -3  # head_dim
