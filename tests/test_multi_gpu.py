"""GPU parity of multi-token decode (a ragged batch of new tokens per sequence,
causal over the cache) against the oracle's float64 definition, on LLaMA- and
Qwen-shaped caches, a sweep of head dims, block sizes, group sizes and query
lengths (pieces of 8 and 16 rows, several pieces per KV head), and bit for bit
against the single-token decode when every sequence has one query."""
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


def queries(w, qlens, seed):
    """Seeded bf16 query rows [sum(qlens), H_q, D] and qo_indptr (int32, device)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    q = torch.randn(int(qo[-1]), w.spec.H_q, w.spec.D, generator=g).to(torch.bfloat16)
    return q.cuda(), qo.cuda()


def run_multi(w, q, qo, max_q_len):
    out = pa.paged_attn_decode_multi(q, w.k_cache, w.v_cache, qo, w.block_tables, w.seq_lens,
                                     w.scale, max_q_len)
    torch.cuda.synchronize()
    return out


def reference(w, q, qo):
    x = oracle.MultiInputs(q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(), w.block_tables.cpu(),
                           w.seq_lens.cpu(), w.scale)
    return oracle.decode_multi(x, qo.cpu())


def assert_parity(out, ref, what=""):
    got = out.float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, \
        f"{what}: max {err.max():.3e} mean {err.mean():.3e}"


@pytest.mark.parametrize("name,qlen", [("llama8b", 4), ("llama8b", 2), ("qwen100k", 3),
                                       ("gqa8", 2), ("tiny", 5)])
def test_published_workloads_multi(name, qlen):
    w = workloads.make(name, device="cuda", poison="nan")
    qlens = [min(qlen, L) for L in w.lens_list]
    q, qo = queries(w, qlens, 7)
    assert_parity(run_multi(w, q, qo, qlen), reference(w, q, qo), f"{name} q_len {qlen}")


def test_one_query_per_sequence_equals_the_decode():
    w = workloads.make("ragged256", device="cuda", poison="nan")
    qlens = [1 if L > 0 else 0 for L in w.lens_list]
    q, qo = queries(w, qlens, 8)
    out = run_multi(w, q, qo, 1)
    # the decode of the same query rows (one per sequence with a token)
    full = torch.zeros_like(w.q)
    idx = torch.tensor([s for s, L in enumerate(w.lens_list) if L > 0], device="cuda")
    full[idx] = q
    dec = pa.paged_attn_decode(full, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), dec[idx].view(torch.int16))


LENS = [1, 15, 16, 17, 31, 33, 100, 257, 1000, 0, 64]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("H_q,H_kv,qmax", [(4, 4, 3), (8, 2, 2), (8, 2, 6), (16, 2, 5),
                                           (16, 1, 1), (6, 1, 7)])
def test_multi_shapes_and_query_lengths(D, BS, H_q, H_kv, qmax):
    sp = workloads.custom_spec("msweep", len(LENS), H_q, H_kv, D, BS, LENS, max_len=1024)
    w = workloads.make(sp, seed=D + BS + H_q + qmax, device="cuda", poison="nan")
    rng = np.random.default_rng(D * BS + qmax)
    qlens = [int(min(L, rng.integers(0, qmax + 1))) for L in LENS]
    qlens[0] = min(LENS[0], qmax)
    q, qo = queries(w, qlens, D + qmax)
    assert_parity(run_multi(w, q, qo, qmax), reference(w, q, qo),
                  f"D{D} BS{BS} G{H_q // H_kv} qmax{qmax}")


def test_multi_long_sequence_split_over_all_ctas():
    sp = workloads.custom_spec("one", 2, 8, 1, 128, 16, [60000, 3000])
    w = workloads.make(sp, seed=3, device="cuda")
    q, qo = queries(w, [4, 4], 9)
    assert_parity(run_multi(w, q, qo, 4), reference(w, q, qo))


def test_multi_repeat_calls_are_bitwise_identical():
    w = workloads.make("llama8b", device="cuda", poison="nan")
    q, qo = queries(w, [3] * w.spec.num_seqs, 10)
    a = run_multi(w, q, qo, 3).clone()
    b = run_multi(w, q, qo, 3)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_multi_rejects_bad_arguments():
    w = workloads.make("tiny", device="cuda")
    q, qo = queries(w, [2, 2], 11)
    lib = pa.load()
    args = [q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(), q.data_ptr(),
            qo.data_ptr(), w.block_tables.data_ptr(), w.seq_lens.data_ptr(), 2, 4]
    tail = [w.spec.H_q, w.spec.H_kv, w.spec.D, int(w.block_tables.shape[1]),
            w.spec.block_size, 0.125, 0]
    assert lib.paged_attn_decode_multi(*args, 0, *tail) == -5          # max_q_len < 1
    assert lib.paged_attn_decode_multi(*args, 200, *tail) == -5        # q_len * G > 256
    assert lib.paged_attn_decode_multi(*(args[:4] + [0] + args[5:]), 2, *tail) == -1


def test_multi_more_sequences_than_one_launch_holds():
    """5,000 sequences (more than one launch takes), two row chunks per KV head."""
    lens = list(np.random.default_rng(12).integers(1, 70, size=5000))
    sp = workloads.custom_spec("wide", len(lens), 8, 1, 64, 16, lens, max_len=80)
    w = workloads.make(sp, seed=12, device="cuda", poison="nan")
    qlens = [int(min(3, L)) for L in lens]
    q, qo = queries(w, qlens, 13)
    assert_parity(run_multi(w, q, qo, 3), reference(w, q, qo), "5000 sequences")


def test_queries_that_see_no_token_are_zero():
    """q_len > seq_len: the first q_len - L queries of that sequence see no token
    (zero rows); the others are the decode of the sequence cut at L - q_len + i + 1."""
    sp = workloads.custom_spec("short", 3, 8, 2, 128, 16, [3, 40, 17], max_len=64)
    w = workloads.make(sp, seed=16, device="cuda", poison="nan")
    qlens = [5, 2, 1]  # sequence 0: queries 0 and 1 see nothing
    q, qo = queries(w, qlens, 17)
    out = run_multi(w, q, qo, 5)
    assert torch.count_nonzero(out[0:2]).item() == 0
    rows_s = np.repeat(np.arange(3), qlens)
    rows_i = np.concatenate([np.arange(n) for n in qlens])
    lens = np.array(w.lens_list)[rows_s]
    cut = lens - (np.array(qlens)[rows_s] - rows_i - 1)
    keep = cut > 0
    single = oracle.Inputs(q.cpu()[keep], w.k_cache.cpu(), w.v_cache.cpu(),
                           w.block_tables.cpu()[rows_s[keep]], torch.tensor(cut[keep], dtype=torch.int32),
                           w.scale)
    assert_parity(out[torch.tensor(keep)], oracle.decode(single), "visible rows")


def test_multi_largest_row_count():
    """q_len 64 with G = 4: 256 query rows per KV head, the most one call takes
    (16 pieces of 16 rows, each KV head's pages walked 16 times)."""
    lens = [64, 700, 2000, 90]
    sp = workloads.custom_spec("maxrows", len(lens), 8, 2, 128, 16, lens, max_len=2048)
    w = workloads.make(sp, seed=21, device="cuda", poison="nan")
    qlens = [64, 64, 33, 64]
    q, qo = queries(w, qlens, 22)
    assert_parity(run_multi(w, q, qo, 64), reference(w, q, qo), "256 rows")


# ---------------------------------------------------------------- without the causal mask
# AstrAI's CUDA Kernels page, "Python Wrappers": is_causal True/False.  Without
# the mask every query row of a sequence attends all of its tokens.

def reference_noncausal(w, q, qo):
    x = oracle.MultiInputs(q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(), w.block_tables.cpu(),
                           w.seq_lens.cpu(), w.scale)
    return oracle.decode_multi(x, qo.cpu(), causal=False)


@pytest.mark.parametrize("name,qlen", [("llama8b", 4), ("llama8b", 8), ("qwen100k", 3),
                                       ("gqa8", 2), ("tiny", 5), ("ragged256", 2)])
def test_noncausal_multi_matches_oracle(name, qlen):
    w = workloads.make(name, device="cuda", poison="nan")
    qlens = [min(qlen, L) for L in w.lens_list]
    q, qo = queries(w, qlens, 61)
    out = pa.paged_attn_decode_multi(q, w.k_cache, w.v_cache, qo, w.block_tables, w.seq_lens,
                                     w.scale, qlen, causal=False)
    torch.cuda.synchronize()
    assert_parity(out, reference_noncausal(w, q, qo), f"{name} q_len {qlen} non-causal")


def test_noncausal_rows_equal_the_decode_of_each_query():
    """Without the mask, every query row of a sequence is the single-token decode of
    that query over the whole sequence: bit for bit when each query is decoded
    alone in a batch of the same shape (q_len 1, whose walk is the decode's)."""
    w = workloads.make("llama8b", device="cuda", poison="nan")
    qlens = [3] * len(w.lens_list)
    q, qo = queries(w, qlens, 62)
    out = pa.paged_attn_decode_multi(q, w.k_cache, w.v_cache, qo, w.block_tables, w.seq_lens,
                                     w.scale, 3, causal=False)
    ref = reference_noncausal(w, q, qo)
    for i in range(3):
        qi = q[i::3].contiguous()
        one = torch.arange(len(w.lens_list) + 1, dtype=torch.int32, device="cuda")
        o1 = pa.paged_attn_decode_multi(qi, w.k_cache, w.v_cache, one, w.block_tables,
                                        w.seq_lens, w.scale, 1, causal=False)
        torch.cuda.synchronize()
        assert_parity(o1, ref[i::3], f"query {i}")
    assert_parity(out, ref, "all")


@pytest.mark.parametrize("D,BS,G,qlen", [(64, 16, 2, 9), (128, 32, 4, 5), (256, 16, 6, 3),
                                         (128, 16, 16, 2), (64, 32, 1, 17)])
def test_noncausal_sweep(D, BS, G, qlen):
    lens = [1, 15, 16, 17, 100, 257, 3, 40]
    sp = workloads.custom_spec("nc_sweep", len(lens), 2 * G, 2, D, BS, lens)
    w = workloads.make(sp, seed=63, device="cuda", poison="nan")
    qlens = [min(qlen, L) for L in lens]
    q, qo = queries(w, qlens, 64)
    out = pa.paged_attn_decode_multi(q, w.k_cache, w.v_cache, qo, w.block_tables, w.seq_lens,
                                     w.scale, qlen, causal=False)
    torch.cuda.synchronize()
    assert_parity(out, reference_noncausal(w, q, qo), f"D {D} BS {BS} G {G} q_len {qlen}")
