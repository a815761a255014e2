"""GPU parity: the sm_103a kernels against the FP64 oracle, element by element.

Tolerance (bf16 in, fp32 accumulate, bf16 out): max |gpu - oracle| <= 2e-2 and
mean |gpu - oracle| <= 2e-3 on every workload; outputs must be finite although
every cache row the definition never reads holds NaN.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pa = pytest.importorskip("paged_kv_gqa_decode_gb300")

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_decode_gb300 import build

    build.build()
    pa.load()


def run_gpu(w, **kw):
    out = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale,
                               **kw)
    torch.cuda.synchronize()
    return out


def errors(out, ref):
    got = out.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref)
    return float(err.max()), float(err.mean())


def assert_parity(out, ref, what=""):
    mx, mean = errors(out, ref)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max {mx:.3e} mean {mean:.3e}"


def reference(w):
    return oracle.decode(workloads.host_copy(w))


@pytest.mark.parametrize("name", ["tiny", "llama8b", "qwen100k", "ragged256", "gqa8"])
def test_published_workloads_full_size(name):
    w = workloads.make(name, device="cuda", poison="nan")
    out = run_gpu(w)
    ref = reference(w)
    assert_parity(out, ref, name)


# The "Add Cuda Kernel" tutorial's paged decode cases (D 128, block 16):
# (num_seqs, context, H_q, H_kv); here with shuffled tables and NaN-filled tails.
@pytest.mark.parametrize("num_seqs,ctx,H_q,H_kv",
                         [(1, 32, 2, 1), (1, 128, 16, 8), (2, 64, 4, 2), (4, 128, 16, 8)])
def test_tutorial_decode_cases(num_seqs, ctx, H_q, H_kv):
    sp = workloads.custom_spec("tutorial", num_seqs, H_q, H_kv, 128, 16, [ctx] * num_seqs)
    w = workloads.make(sp, seed=7, device="cuda")
    assert_parity(run_gpu(w), reference(w))


EDGE_LENS = [0, 1, 15, 16, 17, 31, 32, 33, 100, 257, 1000]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (8, 4), (8, 2), (12, 2), (8, 1), (24, 2), (16, 1)])
def test_shapes_and_ragged_tails(D, BS, H_q, H_kv):
    sp = workloads.custom_spec(f"sweep", len(EDGE_LENS), H_q, H_kv, D, BS, EDGE_LENS,
                               max_len=1024)
    w = workloads.make(sp, seed=D * 1000 + BS * 10 + H_q + H_kv, device="cuda")
    out = run_gpu(w)
    ref = reference(w)
    assert_parity(out, ref, f"D{D} BS{BS} G{H_q // H_kv}")
    # an empty sequence gives an exact zero row
    assert torch.count_nonzero(out[0]).item() == 0


def test_one_token_returns_its_v_row_exactly():
    """L = 1: the softmax weight is exactly 1, so out is the token's V row, bit for bit."""
    sp = workloads.custom_spec("one_tok", 40, 8, 2, 128, 16, [1] * 40, max_len=32)
    w = workloads.make(sp, seed=31, device="cuda", poison="nan")
    out = run_gpu(w)
    G = sp.H_q // sp.H_kv
    blocks = w.block_tables[:, 0].long()
    for h in range(sp.H_q):
        v0 = w.v_cache[blocks, h // G, 0, :]  # [num_seqs, D]
        assert torch.equal(out[:, h].view(torch.int16), v0.view(torch.int16)), f"head {h}"


def test_zero_scale_gives_the_mean_of_v():
    """scale = 0: every visible token weighs the same, out = mean of the V rows."""
    lens = [1, 7, 16, 33, 300, 1000]
    sp = workloads.custom_spec("mean", len(lens), 8, 2, 128, 16, lens, max_len=1024)
    w = workloads.make(sp, seed=32, device="cuda", poison="nan")
    out = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, 0.0)
    torch.cuda.synchronize()
    G = sp.H_q // sp.H_kv
    bs = sp.block_size
    ref = np.zeros((len(lens), sp.H_q, sp.D))
    vc = w.v_cache.double().cpu()
    bt = w.block_tables.cpu()
    for s, L in enumerate(lens):
        t = torch.arange(L)
        for g in range(sp.H_kv):
            rows = vc[bt[s, t // bs].long(), g, t % bs, :]
            ref[s, g * G:(g + 1) * G, :] = rows.mean(dim=0).numpy()
    assert_parity(out, ref, "scale 0")


def test_one_million_token_sequence():
    """One sequence of 2^20 tokens (65,536 pages of one KV head) split over every CTA."""
    sp = workloads.custom_spec("1m", 1, 4, 1, 64, 16, [1 << 20])
    w = workloads.make(sp, seed=33, device="cuda", poison="none")
    assert_parity(run_gpu(w), reference(w), "2^20 tokens")


def test_single_long_sequence_splits_across_all_ctas():
    sp = workloads.custom_spec("one", 1, 8, 1, 128, 16, [60000])
    w = workloads.make(sp, seed=3, device="cuda")
    assert_parity(run_gpu(w), reference(w))


def test_many_short_sequences():
    lens = list(np.random.default_rng(4).integers(0, 40, size=700))
    sp = workloads.custom_spec("short", len(lens), 8, 2, 128, 16, lens, max_len=48)
    w = workloads.make(sp, seed=4, device="cuda")
    assert_parity(run_gpu(w), reference(w))


def test_more_sequences_than_one_launch_holds():
    lens = list(np.random.default_rng(5).integers(1, 70, size=5000))
    sp = workloads.custom_spec("wide", len(lens), 4, 1, 64, 16, lens, max_len=80)
    w = workloads.make(sp, seed=5, device="cuda")
    assert_parity(run_gpu(w), reference(w))


def test_all_sequences_empty():
    sp = workloads.custom_spec("empty", 3, 8, 2, 128, 16, [0, 0, 0], max_len=16)
    w = workloads.make(sp, seed=6, device="cuda")
    out = torch.full_like(w.q, float("nan"))
    run_gpu(w, out=out)
    assert torch.count_nonzero(out).item() == 0


def test_empty_batch():
    w = workloads.make("tiny", device="cuda")
    out = pa.paged_attn_decode(w.q[:0], w.k_cache, w.v_cache, w.block_tables[:0],
                               w.seq_lens[:0], w.scale)
    assert out.shape[0] == 0


def test_lengths_beyond_the_table_are_clamped():
    sp = workloads.custom_spec("cap", 2, 8, 2, 128, 16, [64, 50], max_len=64)
    w = workloads.make(sp, seed=8, device="cuda", poison="none")
    ref = reference(w)
    w2 = workloads.Workload(**{**w.__dict__, "seq_lens": w.seq_lens + torch.tensor(
        [100, 0], dtype=torch.int32, device="cuda")})
    assert_parity(run_gpu(w2), ref)


def test_identity_table_and_relabelled_blocks_agree_bitwise():
    w = workloads.make("llama8b", device="cuda", poison="nan")
    base = run_gpu(w)
    pi = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1)).cuda()
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[pi] = w.k_cache
    v2[pi] = w.v_cache
    bt2 = pi[w.block_tables.long()].int()
    out = pa.paged_attn_decode(w.q, k2, v2, bt2, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_repeat_calls_are_bitwise_identical():
    w = workloads.make("ragged256", device="cuda", poison="nan")
    a = run_gpu(w).clone()
    b = run_gpu(w)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_two_copies_of_the_library_in_one_process(tmp_path):
    # Each copy keeps its own per-device state (shared-memory limits, workspace):
    # a launch through one copy must not make the other skip its own setup.
    import shutil

    other = tmp_path / "libpaged_kv_gqa_decode_copy.so"
    shutil.copy(pa.LIB_PATH, other)
    lib2 = pa.load(str(other))
    w = workloads.make("llama8b", device="cuda", poison="nan")
    a = run_gpu(w).clone()  # the first copy sets up this kernel first
    out = torch.empty_like(w.q)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        rc = lib2.paged_attn_decode(*pa._args(w.q, w.k_cache, w.v_cache, out, w.block_tables,
                                              w.seq_lens, w.scale), stream)
        assert rc == 0, lib2.paged_attn_status_string(rc).decode()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), a.view(torch.int16))
    b = run_gpu(w)
    assert torch.equal(b.view(torch.int16), a.view(torch.int16))


def test_caller_workspace_matches_owned_workspace():
    w = workloads.make("qwen100k", device="cuda", poison="nan")
    base = run_gpu(w).clone()
    n = pa.paged_attn_workspace_bytes(4, 24, 4, 256, w.max_blocks_per_seq, 16)
    assert n > 0
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        out = pa.paged_attn_decode_ws(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                      w.scale, ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), base.view(torch.int16))
    with pytest.raises(pa.PagedAttnError):
        pa.paged_attn_decode_ws(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale,
                                ws[: n // 2])


def test_checked_variant_flags_bad_inputs_without_faulting():
    w = workloads.make("tiny", device="cuda", poison="nan")
    ref = reference(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.paged_attn_decode_checked(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                       w.scale, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_parity(out, ref)
    bad_bt = w.block_tables.clone()
    bad_bt[0, 1] = w.num_blocks + 5     # outside the pool: read as zero rows, flagged
    bad_bt[1, 0] = -3
    pa.paged_attn_decode_checked(w.q, w.k_cache, w.v_cache, bad_bt, w.seq_lens, w.scale, status)
    torch.cuda.synchronize()
    assert status.item() & 1
    status.zero_()
    long = w.seq_lens.clone()
    long[1] = w.max_blocks_per_seq * 16 + 9
    out = pa.paged_attn_decode_checked(w.q, w.k_cache, w.v_cache, w.block_tables, long,
                                       w.scale, status)
    torch.cuda.synchronize()
    assert status.item() & 2


def test_runs_on_a_side_stream_and_in_a_cuda_graph():
    w = workloads.make("llama8b", device="cuda", poison="nan")
    ref = run_gpu(w).clone()
    side = torch.cuda.Stream()
    out = torch.empty_like(w.q)
    with torch.cuda.stream(side):
        pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale,
                             out=out)
    side.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    out2 = torch.empty_like(w.q)
    with torch.cuda.graph(g):
        pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale,
                             out=out2)
    for _ in range(3):
        out2.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))


def test_peaked_softmax_rows():
    # keys scaled so one token dominates each row: stresses the running-max rescale
    sp = workloads.custom_spec("peak", 8, 16, 2, 128, 16, [3000] * 8, peaked_k_frac=0.002,
                               peaked_k_gain=16.0)
    w = workloads.make(sp, seed=9, device="cuda")
    assert_parity(run_gpu(w), reference(w))


def test_one_workspace_serves_calls_of_different_sizes():
    specs = ["qwen100k", "ragged256", "tiny", "gqa8", "llama8b"]
    ws_list = [workloads.make(n, device="cuda", poison="nan") for n in specs]
    need = max(pa.paged_attn_workspace_bytes(w.spec.num_seqs, w.spec.H_q, w.spec.H_kv,
                                             w.spec.D, w.max_blocks_per_seq,
                                             w.spec.block_size) for w in ws_list)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    refs = {}
    for rnd in range(2):
        for n, w in zip(specs, ws_list):
            out = pa.paged_attn_decode_ws(w.q, w.k_cache, w.v_cache, w.block_tables,
                                          w.seq_lens, w.scale, ws)
            torch.cuda.synchronize()
            if rnd == 0:
                refs[n] = reference(w)
            assert_parity(out, refs[n], f"{n} round {rnd}")
    del ws_list


def test_workspace_reuse_across_grids_of_one_two_and_three_ctas_per_sm():
    """head_dim 256 with G = 16 runs one CTA per SM, FP8 caches of head_dim 128
    with 16-token pages three, the others two: partial states written by a
    smaller grid must never land where a larger grid's combine counters live (a
    stale counter corrupts the next call's merge)."""
    wide = workloads.make(workloads.custom_spec("g16d256", 4, 32, 2, 256, 16,
                                                [20000, 15000, 9000, 30000]),
                          device="cuda", poison="nan")
    llama = workloads.make("llama8b", device="cuda", poison="nan")
    gqa8 = workloads.make("gqa8", device="cuda", poison="nan")
    f = workloads.to_fp8(workloads.make("llama8b", seed=7, device="cuda", poison="nan"))
    fref = oracle.decode_fp8(oracle.Fp8Inputs(
        f.q.cpu(), f.k8.cpu(), f.v8.cpu(), f.k_scale.cpu(), f.v_scale.cpu(),
        f.block_tables.cpu(), f.seq_lens.cpu(), f.scale))

    def fp8():
        out = pa.paged_attn_decode_fp8(f.q, f.k8, f.v8, f.k_scale, f.v_scale, f.block_tables,
                                       f.seq_lens, f.scale)
        torch.cuda.synchronize()
        return out

    calls = [(lambda: run_gpu(wide), reference(wide)), (lambda: run_gpu(llama), reference(llama)),
             (fp8, fref), (lambda: run_gpu(wide), None), (lambda: run_gpu(gqa8), reference(gqa8)),
             (fp8, fref)]
    calls[3] = (calls[3][0], calls[0][1])
    for rnd in range(2):
        for i, (call, ref) in enumerate(calls):
            assert_parity(call(), ref, f"call {i} round {rnd}")


def _with_flags(flags, fn):
    pa.paged_attn_set_launch_flags(flags)
    try:
        return fn()
    finally:
        pa.paged_attn_set_launch_flags(0)


def test_early_prologue_gives_the_same_bits():
    """With the early-prologue flag the producer runs ahead of the previous
    launch; results must be bit for bit those of the plain launch, including
    the zero rows of empty sequences."""
    lens = list(np.random.default_rng(41).integers(0, 600, size=90))
    lens[3] = lens[17] = 0
    sp = workloads.custom_spec("early", len(lens), 32, 8, 128, 16, lens, max_len=640)
    w = workloads.make(sp, seed=41, device="cuda", poison="nan")
    plain = run_gpu(w).clone()

    def early():
        outs = [torch.full_like(w.q, float("nan")) for _ in range(4)]
        for o in outs:  # back to back: each launch's producer overlaps the previous one
            pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                 w.scale, out=o)
        torch.cuda.synchronize()
        return outs

    for o in _with_flags(pa.FLAG_EARLY_PROLOGUE, early):
        assert torch.equal(o.view(torch.int16), plain.view(torch.int16))


def test_early_prologue_waits_for_a_query_the_previous_launch_writes():
    """A chain out_k = decode(q = out_{k-1}): each launch reads the query the
    launch before it writes, which the early prologue must still wait for."""
    w = workloads.make("llama8b", device="cuda", poison="nan")

    def chain():
        q = w.q
        for _ in range(4):
            q = pa.paged_attn_decode(q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
        torch.cuda.synchronize()
        return q

    plain = chain()
    assert torch.equal(_with_flags(pa.FLAG_EARLY_PROLOGUE, chain).view(torch.int16),
                       plain.view(torch.int16))


def test_unknown_launch_flags_are_rejected():
    lib = pa.load()
    assert lib.paged_attn_set_launch_flags(2) == -10
    assert lib.paged_attn_set_launch_flags(0) == 0


_GROWTH = r"""
import sys, json
sys.path.insert(0, {root!r})
import numpy as np, torch
import oracle, workloads
import paged_kv_gqa_decode_gb300 as pa
pa.load()
wide = workloads.custom_spec("g16d256", 4, 32, 2, 256, 16, [2000, 1500, 900, 3000])
specs = ["tiny", "llama8b", "tiny", wide, "llama8b"]
ws = [workloads.make(sp, device="cuda", poison="nan") for sp in specs]
side = torch.cuda.Stream()
torch.cuda.synchronize()
outs = []
with torch.cuda.stream(side):
    for w in ws:  # the library-owned workspace grows at calls 1 and 3, no host sync
        outs.append(pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                         w.scale))
side.synchronize()
errs = []
for w, o in zip(ws, outs):
    ref = oracle.decode(workloads.host_copy(w))
    got = o.float().cpu().double().numpy()
    e = np.abs(got - ref)
    errs.append([float(e.max()), float(e.mean()), bool(np.isfinite(got).all())])
print("RESULT " + json.dumps(errs))
"""


def test_owned_workspace_grows_in_stream_order():
    """In a fresh process the library-owned workspace grows twice inside one
    stream of back-to-back calls with no host synchronisation: the smaller buffer
    is released in stream order after the calls that use it, and every call's
    output still matches the oracle."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _GROWTH.format(root=root)], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    for mx, mean, finite in json.loads(r.stdout.split("RESULT ", 1)[1]):
        assert finite and mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)


def test_pinned_host_buffers_give_the_same_bits():
    """q, tables, lengths, query offsets, new rows and outputs in pinned host memory
    (read and written by the kernels over the host link) give the bits that
    device buffers give, for every entry point that takes them."""
    def pin(t):
        return t.cpu().pin_memory()

    w = workloads.make("llama8b", seed=71, device="cuda", poison="nan")
    hq, hbt, hsl = pin(w.q), pin(w.block_tables), pin(w.seq_lens)
    dev = pa.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    hout = torch.empty(tuple(w.q.shape), dtype=w.q.dtype).pin_memory()
    pa.paged_attn_decode(hq, w.k_cache, w.v_cache, hbt, hsl, w.scale, out=hout)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu().view(torch.int16), hout.view(torch.int16))
    # FP8 and x-packed caches
    f = workloads.to_fp8(w)
    dev8 = pa.paged_attn_decode_fp8(w.q, f.k8, f.v8, f.k_scale, f.v_scale, w.block_tables,
                                    w.seq_lens, w.scale)
    h8 = torch.empty_like(hout).pin_memory()
    pa.paged_attn_decode_fp8(hq, f.k8, f.v8, f.k_scale, f.v_scale, hbt, hsl, w.scale, out=h8)
    x = workloads.to_xpacked(w)
    devx = pa.paged_attn_decode_xpacked(w.q, x.kx, x.vt, w.block_tables, w.seq_lens, w.scale)
    hx = torch.empty_like(hout).pin_memory()
    pa.paged_attn_decode_xpacked(hq, x.kx, x.vt, hbt, hsl, w.scale, out=hx)
    # multi-token, query offsets on the host too
    qlens = [3] * len(w.lens_list)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    qm = torch.randn(int(qo[-1]), 32, 128, generator=torch.Generator().manual_seed(72)).to(
        torch.bfloat16)
    devm = pa.paged_attn_decode_multi(qm.cuda(), w.k_cache, w.v_cache, qo.cuda(), w.block_tables,
                                      w.seq_lens, w.scale, 3)
    hm = torch.empty(tuple(qm.shape), dtype=qm.dtype).pin_memory()
    pa.paged_attn_decode_multi(qm.pin_memory(), w.k_cache, w.v_cache, qo.pin_memory(), hbt, hsl,
                               w.scale, 3, out=hm)
    torch.cuda.synchronize()
    assert torch.equal(dev8.cpu().view(torch.int16), h8.view(torch.int16))
    assert torch.equal(devx.cpu().view(torch.int16), hx.view(torch.int16))
    assert torch.equal(devm.cpu().view(torch.int16), hm.view(torch.int16))
    # append + decode with the new rows on the host: same rows in the cache, same output
    g = torch.Generator().manual_seed(73)
    kn = torch.randn(32, 8, 128, generator=g).to(torch.bfloat16)
    vn = torch.randn(32, 8, 128, generator=g).to(torch.bfloat16)
    w2 = workloads.make("llama8b", seed=71, device="cuda", poison="nan")
    dev_a = pa.paged_attn_append_decode(w.q, kn.cuda(), vn.cuda(), w.k_cache, w.v_cache,
                                        w.block_tables, w.seq_lens, w.scale)
    h_a = torch.empty_like(hout).pin_memory()
    pa.paged_attn_append_decode(hq, kn.pin_memory(), vn.pin_memory(), w2.k_cache, w2.v_cache,
                                hbt, hsl, w.scale, out=h_a)
    torch.cuda.synchronize()
    assert torch.equal(dev_a.cpu().view(torch.int16), h_a.view(torch.int16))
    assert torch.equal(w.k_cache.view(torch.int16), w2.k_cache.view(torch.int16))
