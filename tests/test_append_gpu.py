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


# ---------------------------------------------------------------- early prologue
# With FLAG_EARLY_PROLOGUE the decode's producer reads the tables and starts its
# page copies before the work ahead of it has finished.  The append-and-decode
# call must not let its own append break that: where the append is a launch of
# its own (many (sequence, KV head) pieces per CTA, e.g. the ragged 256-sequence
# batch) the decode after it is a plain launch; where the append is fused (the
# LLaMA-shaped batch) the new rows are patched in shared memory.

@pytest.mark.parametrize("name", ["ragged256", "llama8b"])
def test_append_decode_with_early_prologue_back_to_back(name):
    """Two append-and-decode steps back to back under the early prologue, each after
    a kernel that writes q (the usual layer loop), against the oracle and bit for
    bit against the same steps with the flag off."""
    results = []
    for flag in (pa.FLAG_EARLY_PROLOGUE, 0):
        w = workloads.make(name, seed=31, device="cuda", poison="nan")
        before = workloads.host_copy(w)
        q0 = w.q.clone()
        k1, v1 = new_rows(w, 32)
        k2, v2 = new_rows(w, 33)
        pa.paged_attn_set_launch_flags(flag)
        try:
            w.q.copy_(q0 * 2)  # the kernel ahead writes q
            o1 = pa.paged_attn_append_decode(w.q, k1, v1, w.k_cache, w.v_cache,
                                             w.block_tables, w.seq_lens, w.scale)
            o1 = o1.clone()
            w.q.copy_(q0)
            o2 = pa.paged_attn_append_decode(w.q, k2, v2, w.k_cache, w.v_cache,
                                             w.block_tables, w.seq_lens, w.scale)
            torch.cuda.synchronize()
        finally:
            pa.paged_attn_set_launch_flags(0)
        results.append((o1, o2, w.k_cache, w.v_cache))
        if flag:
            step1 = oracle.append(before, k1, v1)
            step1.q = oracle.Inputs(q0 * 2, w.k_cache[:1], w.v_cache[:1], w.block_tables,
                                    w.seq_lens, w.scale).q
            assert_parity(o1, oracle.decode(step1), f"{name} first step")
            step2 = oracle.append(step1, k2, v2)
            step2.q = oracle.Inputs(q0, w.k_cache[:1], w.v_cache[:1], w.block_tables,
                                    w.seq_lens, w.scale).q
            assert np.array_equal(cache_bits(w.k_cache), step2.k)
            assert np.array_equal(cache_bits(w.v_cache), step2.v)
            assert_parity(o2, oracle.decode(step2), f"{name} second step")
    for a, b in zip(results[0], results[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------- multi-token append

def multi_rows(w, qlens, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    shape = (int(qo[-1]), w.spec.H_kv, w.spec.D)
    k = torch.randn(shape, generator=g).to(torch.bfloat16)
    v = torch.randn(shape, generator=g).to(torch.bfloat16)
    q = torch.randn(int(qo[-1]), w.spec.H_q, w.spec.D, generator=g).to(torch.bfloat16)
    return q.cuda(), k.cuda(), v.cuda(), qo.cuda()


MULTI_EDGE = workloads.custom_spec("multi_append_edges", 9, 8, 2, 128, 16,
                                   [1, 15, 16, 17, 31, 33, 0, 48, 1000], max_len=1024)


@pytest.mark.parametrize("name,qlen", [("edges", 17), ("llama8b", 4), ("gqa8", 3),
                                       ("qwen100k", 2), ("tiny", 5)])
def test_multi_append_writes_exactly_the_oracle_rows(name, qlen):
    """q_len new rows per sequence (more than a page, and more than some sequences
    hold) land where the oracle puts them, bit for bit, and nothing else moves."""
    w = workloads.make(MULTI_EDGE if name == "edges" else name, seed=34, device="cuda",
                       poison="nan")
    rng = np.random.default_rng(34)
    qlens = [int(rng.integers(0, qlen + 1)) for _ in w.lens_list]
    q, k_new, v_new, qo = multi_rows(w, qlens, 35)
    exp = oracle.append_multi(workloads.host_copy(w), qo.cpu(), k_new.cpu(), v_new.cpu())
    pa.paged_kv_append_multi(k_new, v_new, w.k_cache, w.v_cache, qo, w.block_tables, w.seq_lens)
    torch.cuda.synchronize()
    assert np.array_equal(cache_bits(w.k_cache), exp.k)
    assert np.array_equal(cache_bits(w.v_cache), exp.v)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("name,qlen", [("edges", 17), ("llama8b", 4)])
def test_multi_append_decode_matches_oracle(name, qlen, causal):
    w = workloads.make(MULTI_EDGE if name == "edges" else name, seed=36, device="cuda",
                       poison="nan")
    qlens = [min(qlen, L) for L in w.lens_list]
    q, k_new, v_new, qo = multi_rows(w, qlens, 37)
    exp = oracle.append_multi(workloads.host_copy(w), qo.cpu(), k_new.cpu(), v_new.cpu())
    pa.paged_attn_set_launch_flags(pa.FLAG_EARLY_PROLOGUE)  # must not matter here
    try:
        out = pa.paged_attn_append_decode_multi(q, k_new, v_new, w.k_cache, w.v_cache, qo,
                                                w.block_tables, w.seq_lens, w.scale, qlen,
                                                causal=causal)
        torch.cuda.synchronize()
    finally:
        pa.paged_attn_set_launch_flags(0)
    assert np.array_equal(cache_bits(w.k_cache), exp.k)
    x = oracle.MultiInputs(q.cpu(), exp.k, exp.v, exp.bt, exp.lens, w.scale)
    assert_parity(out, oracle.decode_multi(x, qo.cpu(), causal=causal), f"{name} {causal}")


# ---------------------------------------------------------------- FP8 append

def fp8_bits(f):
    return (f.k8.cpu().numpy(), f.v8.cpu().numpy(), f.k_scale.cpu().numpy(),
            f.v_scale.cpu().numpy())


@pytest.mark.parametrize("name", ["edges", "llama8b", "qwen100k", "ragged256"])
def test_fp8_append_writes_the_oracle_bytes_and_floats(name):
    """Quantize-on-append: the e4m3 bytes and the row floats the kernel writes are
    the oracle's bit for bit (the rounding decision is taken in float32 on both
    sides), and every other byte and float is left as it was."""
    w = workloads.make(EDGE if name == "edges" else name, seed=38, device="cuda", poison="nan")
    f = workloads.to_fp8(w)
    k_new, v_new = new_rows(w, 39)
    k_new[0].zero_()  # an all-zero K row: float 1
    host = oracle.Fp8Inputs(f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(),
                            f.v_scale.cpu(), f.block_tables.cpu(), f.seq_lens.cpu(), f.scale)
    exp = oracle.append_fp8(host, k_new.cpu(), v_new.cpu())
    pa.paged_kv_append_fp8(k_new, v_new, f.k8, f.v8, f.k_scale, f.v_scale, f.block_tables,
                           f.seq_lens)
    torch.cuda.synchronize()
    k8, v8, ks, vs = fp8_bits(f)
    assert np.array_equal(k8, exp.k8) and np.array_equal(v8, exp.v8)
    # floats compared as bit patterns (NaN floats of unread rows included)
    assert np.array_equal(ks.view(np.uint32), exp.ks.view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), exp.vs.view(np.uint32))


@pytest.mark.parametrize("name", ["edges", "llama8b", "ragged256"])
def test_fp8_append_decode_matches_oracle(name):
    w = workloads.make(EDGE if name == "edges" else name, seed=40, device="cuda", poison="nan")
    f = workloads.to_fp8(w)
    k_new, v_new = new_rows(w, 41)
    host = oracle.Fp8Inputs(f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(),
                            f.v_scale.cpu(), f.block_tables.cpu(), f.seq_lens.cpu(), f.scale)
    exp = oracle.append_fp8(host, k_new.cpu(), v_new.cpu())
    pa.paged_attn_set_launch_flags(pa.FLAG_EARLY_PROLOGUE)  # must not matter here
    try:
        out = pa.paged_attn_append_decode_fp8(f.q, k_new, v_new, f.k8, f.v8, f.k_scale,
                                              f.v_scale, f.block_tables, f.seq_lens, f.scale)
        torch.cuda.synchronize()
    finally:
        pa.paged_attn_set_launch_flags(0)
    assert np.array_equal(f.k8.cpu().numpy(), exp.k8)
    assert_parity(out, oracle.decode_fp8(exp), name)


@pytest.mark.parametrize("name", ["edges", "llama8b"])
def test_fused_fp8_append_decode_equals_append_then_decode(name):
    """The fused FP8 append (quantized in the decode's shared memory) writes the
    bytes and floats the standalone append writes and gives the same output bits
    as the standalone append followed by the decode."""
    sp = EDGE if name == "edges" else workloads.spec(name)
    res = []
    for fused in (True, False):
        w = workloads.make(sp, seed=42, device="cuda", poison="nan")
        f = workloads.to_fp8(w)
        k_new, v_new = new_rows(w, 43)
        if fused:
            out = pa.paged_attn_append_decode_fp8(f.q, k_new, v_new, f.k8, f.v8, f.k_scale,
                                                  f.v_scale, f.block_tables, f.seq_lens, f.scale)
        else:
            pa.paged_kv_append_fp8(k_new, v_new, f.k8, f.v8, f.k_scale, f.v_scale,
                                   f.block_tables, f.seq_lens)
            out = pa.paged_attn_decode_fp8(f.q, f.k8, f.v8, f.k_scale, f.v_scale, f.block_tables,
                                           f.seq_lens, f.scale)
        torch.cuda.synchronize()
        res.append((out, f.k8, f.v8, f.k_scale.view(torch.int32), f.v_scale.view(torch.int32)))
    for a, b in zip(*res):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_fused_fp8_append_decode_with_early_prologue_back_to_back():
    """Two fused FP8 append-decode steps under the early prologue, each after a
    kernel that writes q, against the oracle (the fused branch: LLaMA shape)."""
    w = workloads.make("llama8b", seed=44, device="cuda", poison="nan")
    f = workloads.to_fp8(w)
    host = oracle.Fp8Inputs(f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(),
                            f.v_scale.cpu(), f.block_tables.cpu(), f.seq_lens.cpu(), f.scale)
    q0 = f.q.clone()
    k1, v1 = new_rows(w, 45)
    k2, v2 = new_rows(w, 46)
    pa.paged_attn_set_launch_flags(pa.FLAG_EARLY_PROLOGUE)
    try:
        w.q.copy_(q0 * 2)
        o1 = pa.paged_attn_append_decode_fp8(w.q, k1, v1, f.k8, f.v8, f.k_scale, f.v_scale,
                                             f.block_tables, f.seq_lens, f.scale).clone()
        w.q.copy_(q0)
        o2 = pa.paged_attn_append_decode_fp8(w.q, k2, v2, f.k8, f.v8, f.k_scale, f.v_scale,
                                             f.block_tables, f.seq_lens, f.scale)
        torch.cuda.synchronize()
    finally:
        pa.paged_attn_set_launch_flags(0)
    step1 = oracle.append_fp8(host, k1.cpu(), v1.cpu())
    step1.q = oracle.Inputs(q0 * 2, w.k_cache[:1], w.v_cache[:1], w.block_tables, w.seq_lens,
                            w.scale).q
    assert_parity(o1, oracle.decode_fp8(step1), "first step")
    step2 = oracle.append_fp8(step1, k2.cpu(), v2.cpu())
    step2.q = oracle.Inputs(q0, w.k_cache[:1], w.v_cache[:1], w.block_tables, w.seq_lens,
                            w.scale).q
    assert np.array_equal(f.k8.cpu().numpy(), step2.k8)
    assert np.array_equal(f.v_scale.cpu().numpy().view(np.uint32), step2.vs.view(np.uint32))
    assert_parity(o2, oracle.decode_fp8(step2), "second step")
