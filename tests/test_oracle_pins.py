"""Pins for the FP64 oracle: each test ties it to something other than itself.

* a library routine: torch's float64 scaled_dot_product_attention on the
  contiguous (un-paged) K/V that the test pages itself;
* closed forms: one token, constant V rows, zero query / zero scale, and a
  hand-worked example stored under tests/golden/;
* invariances: relabelling physical blocks, duplicating KV heads, NaN in every
  row the definition never reads, scores large enough that exp overflows
  without the max shift;
* the split/merge algebra of the split-KV design: merging the pieces of any
  partition of [0, L) equals the whole-sequence result.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _page(K, V, BS, gen_np, extra_blocks=1, fill=float("nan")):
    """Scatter contiguous per-sequence K/V ([L_s, H_kv, D] each) into a shuffled pool.

    Returns (k_cache, v_cache, block_tables, seq_lens); unused rows hold ``fill``.
    """
    H_kv, D = K[0].shape[1], K[0].shape[2]
    lens = [k.shape[0] for k in K]
    pages = [-(-L // BS) for L in lens]
    maxb = max(1, max(pages))
    nb = sum(pages) + extra_blocks
    perm = gen_np.permutation(nb)
    kc = torch.full((nb, H_kv, BS, D), fill, dtype=torch.bfloat16)
    vc = torch.full((nb, H_kv, BS, D), fill, dtype=torch.bfloat16)
    bt = np.full((len(K), maxb), perm[-1], dtype=np.int32)
    pos = 0
    for s, L in enumerate(lens):
        for p in range(pages[s]):
            b = int(perm[pos])
            pos += 1
            bt[s, p] = b
            t0, t1 = p * BS, min(L, (p + 1) * BS)
            # cache row order is [block, head, slot, dim]; contiguous is [token, head, dim]
            kc[b, :, : t1 - t0, :] = K[s][t0:t1].transpose(0, 1)
            vc[b, :, : t1 - t0, :] = V[s][t0:t1].transpose(0, 1)
    return kc, vc, torch.from_numpy(bt), torch.tensor(lens, dtype=torch.int32)


def _sdpa(q, K, V, scale):
    """torch float64 SDPA per sequence on contiguous K/V, GQA by repeating KV heads."""
    outs = []
    H_q = q.shape[1]
    for s in range(q.shape[0]):
        k = K[s].double().transpose(0, 1)  # [H_kv, L, D]
        v = V[s].double().transpose(0, 1)
        G = H_q // k.shape[0]
        k = k.repeat_interleave(G, dim=0)[None]
        v = v.repeat_interleave(G, dim=0)[None]
        qq = q[s].double()[None, :, None, :]  # [1, H_q, 1, D]
        outs.append(F.scaled_dot_product_attention(qq, k, v, scale=scale)[0, :, 0, :])
    return torch.stack(outs).numpy()


def _random_problem(seed, lens, H_q, H_kv, D, BS, kv_std=1.0, extra_blocks=1):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    q = _bf16(torch.randn(len(lens), H_q, D, generator=g))
    K = [_bf16(torch.randn(L, H_kv, D, generator=g) * kv_std) for L in lens]
    V = [_bf16(torch.randn(L, H_kv, D, generator=g) * kv_std) for L in lens]
    kc, vc, bt, sl = _page(K, V, BS, rng, extra_blocks=extra_blocks)
    return q, K, V, kc, vc, bt, sl


CASES = [
    # seed, lens, H_q, H_kv, D, BS
    (1, [37, 100], 4, 2, 64, 16),
    (2, [1, 16, 17, 33], 8, 8, 32, 16),     # G = 1 (plain multi-head)
    (3, [5, 64, 129], 6, 1, 128, 32),        # G = 6
    (4, [31, 2, 48], 16, 2, 16, 8),          # G = 8
    (5, [200], 3, 1, 8, 4),                  # odd sizes the definition allows
]


@pytest.mark.parametrize("seed,lens,H_q,H_kv,D,BS", CASES)
def test_matches_torch_sdpa_on_unpaged_kv(seed, lens, H_q, H_kv, D, BS):
    q, K, V, kc, vc, bt, sl = _random_problem(seed, lens, H_q, H_kv, D, BS)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    got = oracle.decode(oracle.Inputs(q, kc, vc, bt, sl, scale))
    ref = _sdpa(q, K, V, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_golden_worked_example():
    with open(os.path.join(GOLDEN, "paged_decode_worked_example.json")) as f:
        ex = json.load(f)
    nb, H_kv, BS, D = ex["num_blocks"], ex["H_kv"], ex["block_size"], ex["D"]
    kc = torch.full((nb, H_kv, BS, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    for r in ex["k_rows"]:
        kc[r["block"], r["head"], r["slot"]] = torch.tensor(r["values"], dtype=torch.bfloat16)
    for r in ex["v_rows"]:
        vc[r["block"], r["head"], r["slot"]] = torch.tensor(r["values"], dtype=torch.bfloat16)
    q = torch.tensor(ex["q"], dtype=torch.bfloat16)
    bt = torch.tensor(ex["block_tables"], dtype=torch.int32)
    sl = torch.tensor(ex["seq_lens"], dtype=torch.int32)
    got = oracle.decode(oracle.Inputs(q, kc, vc, bt, sl, ex["scale"]))

    def value(expr):
        # the fixture's closed forms use numbers, e, + - * / and parentheses only
        if not set(expr) <= set("0123456789.e+-*/() "):
            raise ValueError(expr)
        return float(eval(expr, {"__builtins__": {}}, {"e": math.e}))

    for row in ex["expected"]:
        want = np.array([value(v) for v in row["values"]])
        np.testing.assert_allclose(got[row["s"], row["h"]], want, rtol=0,
                                   atol=ex["abs_tolerance"])


def test_single_token_returns_its_v_row():
    q, K, V, kc, vc, bt, sl = _random_problem(11, [1, 1, 1], 4, 2, 64, 16)
    got = oracle.decode(oracle.Inputs(q, kc, vc, bt, sl, 0.125))
    for s in range(3):
        for h in range(4):
            want = V[s][0, h // 2].double().numpy()
            assert np.array_equal(got[s, h], want)


def test_constant_v_rows_return_the_constant():
    lens = [3, 50, 97]
    q, K, V, kc, vc, bt, sl = _random_problem(12, lens, 4, 2, 32, 16)
    c = _bf16(torch.randn(2, 32, generator=torch.Generator().manual_seed(5)))
    V = [c[None].expand(L, 2, 32).clone() for L in lens]
    kc2, vc2, bt2, sl2 = _page(K, V, 16, np.random.default_rng(12))
    got = oracle.decode(oracle.Inputs(q, kc2, vc2, bt2, sl2, 0.3))
    for s in range(3):
        for h in range(4):
            np.testing.assert_allclose(got[s, h], c[h // 2].double().numpy(), rtol=1e-15,
                                       atol=1e-15)


@pytest.mark.parametrize("zero", ["query", "scale"])
def test_uniform_weights_give_the_mean_of_v(zero):
    lens = [7, 40, 129]
    q, K, V, kc, vc, bt, sl = _random_problem(13, lens, 6, 3, 64, 16)
    scale = 0.125
    if zero == "query":
        q = torch.zeros_like(q)
    else:
        scale = 0.0
    got = oracle.decode(oracle.Inputs(q, kc, vc, bt, sl, scale))
    for s, L in enumerate(lens):
        mean = V[s].double().mean(dim=0).numpy()  # [H_kv, D]
        for h in range(6):
            np.testing.assert_allclose(got[s, h], mean[h // 2], rtol=0, atol=1e-14)


def test_block_relabelling_is_invisible():
    w = workloads.make("tiny", poison="nan")
    base = oracle.decode(w)
    rng = np.random.default_rng(99)
    pi = rng.permutation(w.num_blocks)               # old id -> new id
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[torch.from_numpy(pi)] = w.k_cache
    v2[torch.from_numpy(pi)] = w.v_cache
    bt2 = torch.from_numpy(pi[w.block_tables.numpy()].astype(np.int32))
    got = oracle.decode(oracle.Inputs(w.q, k2, v2, bt2, w.seq_lens, w.scale))
    assert np.array_equal(got, base)


def test_duplicated_kv_heads_give_the_same_rows():
    w = workloads.make("tiny", poison="nan")
    G = w.spec.G
    base = oracle.decode(w)
    # one KV head per query head, holding the KV head that query head maps to
    k2 = w.k_cache.repeat_interleave(G, dim=1)
    v2 = w.v_cache.repeat_interleave(G, dim=1)
    got = oracle.decode(oracle.Inputs(w.q, k2, v2, w.block_tables, w.seq_lens, w.scale))
    assert np.array_equal(got, base)


def test_unread_rows_never_matter():
    clean = workloads.make("tiny", poison="none")
    poisoned = workloads.make("tiny", poison="nan")
    a = oracle.decode(clean)
    b = oracle.decode(poisoned)
    assert np.isfinite(b).all()
    assert np.array_equal(a, b)


def test_large_scores_stay_finite_and_exact():
    # scores near 1e3 overflow exp() unless the row max is subtracted first
    q, K, V, kc, vc, bt, sl = _random_problem(14, [20, 70], 2, 1, 64, 16, kv_std=16.0)
    q = q * 16
    scale = 1.0
    got = oracle.decode(oracle.Inputs(q, kc, vc, bt, sl, scale))
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, _sdpa(q, K, V, scale), rtol=0, atol=1e-12)


def _random_partition(rng, L, parts):
    cuts = np.sort(rng.integers(0, L + 1, size=parts - 1))
    edges = [0] + [int(c) for c in cuts] + [L]
    return list(zip(edges[:-1], edges[1:]))  # may contain empty and singleton ranges


@pytest.mark.parametrize("parts", [1, 2, 5, 17])
def test_merging_partition_pieces_equals_whole(parts):
    w = workloads.make("tiny", poison="nan")
    inp = oracle.Inputs.from_workload(w)
    whole = oracle.decode(inp)
    rng = np.random.default_rng(parts)
    for s, L in enumerate(w.lens_list):
        for h in range(w.spec.H_q):
            rngs = _random_partition(rng, L, parts)
            M, l, o = oracle.pieces(inp, [(s, h)] * len(rngs), rngs)
            order = rng.permutation(len(rngs))  # the merge is order-free
            state = (-np.inf, 0.0, np.zeros(w.spec.D))
            for i in order:
                state = oracle.combine(state, (M[i], l[i], o[i]))
            np.testing.assert_allclose(oracle.finish(state), whole[s, h], rtol=1e-13, atol=1e-15)


def test_combine_is_associative_and_commutative():
    rng = np.random.default_rng(3)
    st = [(float(rng.normal() * 5), float(rng.uniform(0.5, 9)), rng.normal(size=8))
          for _ in range(3)]
    a, b, c = st
    ab_c = oracle.combine(oracle.combine(a, b), c)
    a_bc = oracle.combine(a, oracle.combine(b, c))
    assert ab_c[0] == a_bc[0]
    np.testing.assert_allclose(ab_c[1], a_bc[1], rtol=1e-14)
    np.testing.assert_allclose(ab_c[2], a_bc[2], rtol=1e-14)
    ba = oracle.combine(b, a)
    ab = oracle.combine(a, b)
    assert ab[0] == ba[0] and ab[1] == ba[1] and np.array_equal(ab[2], ba[2])
    empty = (-np.inf, 0.0, np.zeros(8))
    e_a = oracle.combine(empty, a)
    assert e_a[0] == a[0] and e_a[1] == a[1] and np.array_equal(e_a[2], a[2])


def test_empty_sequence_gives_zero_row():
    # the pages do not define an empty softmax; the documented reading is a zero row
    q, K, V, kc, vc, bt, sl = _random_problem(15, [0, 9], 2, 1, 16, 8)
    got = oracle.decode(oracle.Inputs(q, kc, vc, bt, sl, 0.25))
    assert np.array_equal(got[0], np.zeros((2, 16)))
    assert np.isfinite(got[1]).all()


def test_rows_subset_matches_full():
    w = workloads.make("tiny", poison="nan")
    full = oracle.decode(w)
    pairs = [(1, 3), (0, 0), (1, 0)]
    sub = oracle.decode(w, pairs=pairs)
    for i, (s, h) in enumerate(pairs):
        assert np.array_equal(sub[i], full[s, h])


def test_bad_inputs_are_rejected():
    w = workloads.make("tiny", poison="nan")
    inp = oracle.Inputs.from_workload(w)
    bad_bt = w.block_tables.clone()
    bad_bt[0, 0] = w.num_blocks
    with pytest.raises(oracle.OracleError):
        oracle.decode(oracle.Inputs(w.q, w.k_cache, w.v_cache, bad_bt, w.seq_lens, w.scale))
    long = w.seq_lens.clone()
    long[0] = inp.maxb * inp.BS + 1
    with pytest.raises(oracle.OracleError):
        oracle.decode(oracle.Inputs(w.q, w.k_cache, w.v_cache, w.block_tables, long, w.scale))
    q3 = torch.zeros(2, 3, 64, dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.decode(oracle.Inputs(q3, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, 0.1))


MUTANTS = [
    ("kv head h % H_kv", "(int)(((long long)h * H_kv) / H_q)", "(h % H_kv)"),
    ("scale dropped", "z[t - t0] = scale * dot;", "z[t - t0] = dot;"),
    ("page index from t % BS", "bt[(size_t)s * max_blocks + t / BS]", "bt[(size_t)s * max_blocks + t % BS]"),
    ("slot index from t / BS", "(pb * H_kv + g) * BS + (size_t)(t % BS);",
     "(pb * H_kv + g) * BS + (size_t)(t / BS);"),
    ("max not subtracted", "exp(z[t - t0] - M)", "exp(z[t - t0])"),
    ("softmax sign flipped", "exp(z[t - t0] - M)", "exp(M - z[t - t0])"),
    ("last token dropped", "for (int t = t0; t < t1; ++t) {\n        const double w",
     "for (int t = t0; t < t1 - 1; ++t) {\n        const double w"),
    ("no normalisation", "out_row[d] /= l;", "out_row[d] /= 1.0;"),
    ("K row reversed", "widen_bf16(qrow[d]) * cache_k(c, krow, d, D)",
     "widen_bf16(qrow[d]) * cache_k(c, krow, D - 1 - d, D)"),
    ("query head from kv head", "qrow = q + ((size_t)s * H_q + h) * D",
     "qrow = q + ((size_t)s * H_q + g) * D"),
]


def _pins_pass() -> bool:
    """The cheap pins, run against whatever library oracle._lib holds."""
    try:
        test_matches_torch_sdpa_on_unpaged_kv(*CASES[0])
        test_matches_torch_sdpa_on_unpaged_kv(*CASES[3])
        test_golden_worked_example()
        test_single_token_returns_its_v_row()
        test_unread_rows_never_matter()
        test_large_scores_stay_finite_and_exact()
        test_merging_partition_pieces_equals_whole(5)
    except (AssertionError, oracle.OracleError, FloatingPointError):
        return False
    return True


_MUTANT_RUNNER = """
import ctypes, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import oracle
import test_oracle_pins as T
good = oracle._load()
lib = ctypes.CDLL({so!r})
for fn in ("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs"):
    getattr(lib, fn).argtypes = getattr(good, fn).argtypes
    getattr(lib, fn).restype = getattr(good, fn).restype
oracle._lib = lib
with np.errstate(all="ignore"):
    print("PINS_PASS" if T._pins_pass() else "PINS_FAIL")
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(name, old, new, tmp_path):
    """Plant a plausible mistake in a copy of the oracle's C source, build it, and check
    that at least one pin fails against the mutant (run in a child process, since a
    mutant may also read out of bounds and crash, which counts as caught)."""
    import subprocess
    import sys

    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutant), "-lm"], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = _MUTANT_RUNNER.format(root=os.path.dirname(here), tests=here, so=str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    crashed = r.returncode < 0  # killed by a signal: the mutant read out of bounds
    assert crashed or "PINS_FAIL" in r.stdout, \
        f"no pin noticed the planted mistake: {name}\n{r.stdout}\n{r.stderr[-2000:]}"


def test_unmutated_oracle_passes_the_same_pins():
    assert _pins_pass()


# ---------------------------------------------------------------- cache append

def _last_rows(inp):
    """Each sequence's newest cached K and V rows, [num_seqs, H_kv, D] (zeros when L = 0).

    Read through the un-paged view (the table maps logical page i of s to its block),
    so these tests do not restate the append's own indexing."""
    k = np.zeros((inp.num_seqs, inp.H_kv, inp.D), dtype=np.uint16)
    v = np.zeros_like(k)
    for s in range(inp.num_seqs):
        L = int(inp.lens[s])
        if L == 0:
            continue
        pages = [inp.bt[s, i] for i in range(-(-L // inp.BS))]
        flat_k = np.concatenate([inp.k[b] for b in pages], axis=1)  # [H_kv, pages*BS, D]
        flat_v = np.concatenate([inp.v[b] for b in pages], axis=1)
        k[s] = flat_k[:, L - 1]
        v[s] = flat_v[:, L - 1]
    return k, v


def _append_pins_pass(append) -> bool:
    """The cache-append pins, against a given append function."""
    try:
        _round_trip(append, "tiny")
        _round_trip(append, "ragged_small")
        test_append_changes_only_the_new_token_rows(append)
        test_append_of_a_one_token_sequence_is_its_output(append)
    except (AssertionError, oracle.OracleError, IndexError, ValueError):
        return False
    return True


@pytest.fixture
def append():
    return oracle.append


@pytest.mark.parametrize("name", ["tiny", "ragged_small"])
def test_append_round_trip_restores_cache_and_decode(append, name):
    _round_trip(append, name)


def _round_trip(append, name):
    """Take every sequence's newest row out of the cache, poison it, append it back:
    the caches and the decode come back bit for bit."""
    if name == "ragged_small":
        spec = workloads.custom_spec("ragged_small", 9, 8, 2, 64, 16,
                                     [1, 15, 16, 17, 31, 32, 33, 0, 48])
        w = workloads.make(spec, seed=7, poison="nan")
    else:
        w = workloads.make(name, poison="nan")
    inp = oracle.Inputs.from_workload(w)
    k_new, v_new = _last_rows(inp)
    hole = oracle.Inputs.from_workload(w)
    hole.k, hole.v = hole.k.copy(), hole.v.copy()  # the views share the workload's memory
    for s in range(hole.num_seqs):  # poison the newest row of every sequence
        L = int(hole.lens[s])
        if L == 0:
            continue
        pages = -(-L // hole.BS)
        b = int(hole.bt[s, pages - 1])
        slot = (L - 1) - (pages - 1) * hole.BS
        hole.k[b, :, slot, :] = 0x7FC0
        hole.v[b, :, slot, :] = 0x7FC0
    back = append(hole, k_new, v_new)
    assert np.array_equal(back.k, inp.k) and np.array_equal(back.v, inp.v)
    assert np.array_equal(oracle.decode(back), oracle.decode(inp))


def test_append_changes_only_the_new_token_rows(append):
    """Random new rows: exactly H_kv * D values per non-empty sequence change in each cache,
    and the input problem itself is left untouched."""
    spec = workloads.custom_spec("app", 5, 4, 2, 64, 16, [3, 16, 0, 17, 40])
    w = workloads.make(spec, seed=11, poison="zero")
    inp = oracle.Inputs.from_workload(w)
    k0, v0 = inp.k.copy(), inp.v.copy()
    rng = np.random.default_rng(3)
    # magnitudes 32768..65535, which the N(0, 1) cache never holds: every written value changes
    k_new = rng.integers(0x4700, 0x4780, size=(5, 2, 64), dtype=np.uint16)
    v_new = rng.integers(0xC700, 0xC780, size=(5, 2, 64), dtype=np.uint16)
    out = append(inp, k_new, v_new)
    assert np.array_equal(inp.k, k0) and np.array_equal(inp.v, v0)
    nonempty = sum(1 for L in [3, 16, 0, 17, 40] if L > 0)
    assert int((out.k != k0).sum()) == nonempty * 2 * 64
    assert int((out.v != v0).sum()) == nonempty * 2 * 64
    kl, vl = _last_rows(out)
    for s, L in enumerate([3, 16, 0, 17, 40]):
        if L:
            assert np.array_equal(kl[s], k_new[s]) and np.array_equal(vl[s], v_new[s])


def test_append_of_a_one_token_sequence_is_its_output(append):
    """A sequence whose only token is the new one attends to it alone: out = v_new."""
    spec = workloads.custom_spec("one", 3, 4, 2, 64, 16, [1, 1, 1])
    w = workloads.make(spec, seed=5, poison="nan")
    rng = np.random.default_rng(9)
    k_new = rng.integers(0x3C00, 0x4000, size=(3, 2, 64), dtype=np.uint16)
    v_new = rng.integers(0x3C00, 0x4000, size=(3, 2, 64), dtype=np.uint16)
    out = oracle.decode(append(oracle.Inputs.from_workload(w), k_new, v_new))
    vf = (v_new.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(out[s, h], vf[s, h // 2])


APPEND_MUTANTS = [
    ("slot from L", "t % inp.BS, :] = kn[s]", "L % inp.BS, :] = kn[s]"),
    ("page from L", "b = int(inp.bt[s, t // inp.BS])", "b = int(inp.bt[s, L // inp.BS])"),
    ("k and v swapped", "out.v[b, :, t % inp.BS, :] = vn[s]", "out.v[b, :, t % inp.BS, :] = kn[s]"),
    ("kv head dropped", "out.k[b, :, t % inp.BS, :] = kn[s]", "out.k[b, :, t % inp.BS, :] = kn[s, 0]"),
]


@pytest.mark.parametrize("name,old,new", APPEND_MUTANTS, ids=[m[0] for m in APPEND_MUTANTS])
def test_append_pins_catch_planted_mistakes(name, old, new):
    import inspect

    src = inspect.getsource(oracle.append)
    assert src.count(old) == 1, name
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    assert not _append_pins_pass(ns["append"]), f"no pin noticed: {name}"


def test_unmutated_append_passes_the_same_pins():
    assert _append_pins_pass(oracle.append)


# ---------------------------------------------------------------- FP8 caches

def test_e4m3_decoding_matches_torch_float8():
    """Every byte code decodes as torch's float8_e4m3fn does (NaN codes included)."""
    t = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(t), np.isnan(ref))
    assert np.array_equal(t[~np.isnan(t)], ref[~np.isnan(ref)])


def _fp8_with_exact_bf16_twin(seed=0, lens=(1, 15, 16, 17, 40), H_q=8, H_kv=2, D=64, BS=16):
    """An FP8 problem with random finite e4m3 codes and power-of-two row floats,
    and the bf16 problem holding exactly the same values (e4m3 x 2^k is exact in
    bf16), built without the oracle's decoder: through torch's float8 type."""
    spec = workloads.custom_spec("fp8twin", len(lens), H_q, H_kv, D, BS, list(lens))
    w = workloads.make(spec, seed=seed, poison="none")
    rng = np.random.default_rng(seed)
    shape = tuple(w.k_cache.shape)
    codes = rng.integers(0, 256, size=(2,) + shape, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38  # no NaN codes (0x38 = 1.0)
    scales = np.ldexp(1.0, rng.integers(-6, 7, size=(2,) + shape[:3])).astype(np.float32)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double() * \
        torch.from_numpy(scales).double().unsqueeze(-1)
    k16, v16 = vals[0].to(torch.bfloat16), vals[1].to(torch.bfloat16)
    assert torch.equal(k16.double(), vals[0]) and torch.equal(v16.double(), vals[1])
    bf = oracle.Inputs(w.q, k16, v16, w.block_tables, w.seq_lens, w.scale)
    f8 = oracle.Fp8Inputs(w.q, codes[0], codes[1], scales[0], scales[1], w.block_tables,
                          w.seq_lens, w.scale)
    return f8, bf


def test_fp8_decode_equals_bf16_decode_of_the_same_values():
    for seed in range(3):
        f8, bf = _fp8_with_exact_bf16_twin(seed)
        assert np.array_equal(oracle.decode_fp8(f8), oracle.decode(bf))


def test_fp8_row_floats_scale_as_stated():
    f8, _ = _fp8_with_exact_bf16_twin(7)
    base = oracle.decode_fp8(f8)
    f8.vs = f8.vs * np.float32(4.0)        # every V row x4: the output x4
    assert np.allclose(oracle.decode_fp8(f8), 4.0 * base, rtol=1e-12, atol=0)
    f8.vs = f8.vs / np.float32(4.0)
    f8.ks = f8.ks * np.float32(2.0)        # every K row x2 == softmax scale x2
    twice = oracle.decode_fp8(f8)
    f8.ks = f8.ks / np.float32(2.0)
    f8.scale = float(np.float32(2.0 * f8.scale))
    assert np.allclose(twice, oracle.decode_fp8(f8), rtol=1e-12, atol=1e-15)


def _fp8_pins_pass() -> bool:
    try:
        test_e4m3_decoding_matches_torch_float8()
        test_fp8_decode_equals_bf16_decode_of_the_same_values()
        test_fp8_row_floats_scale_as_stated()
    except (AssertionError, oracle.OracleError, FloatingPointError):
        return False
    return True


FP8_MUTANTS = [
    ("exponent bias 8", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("subnormal scale", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    ("sign dropped", "return sign ? -v : v;", "return v;"),
    ("K row float from V", "* (double)c->k_scale[row];", "* (double)c->v_scale[row];"),
    ("row float of the next row", "* (double)c->v_scale[row];", "* (double)c->v_scale[row + 1];"),
    ("mantissa 4 bits", "(double)m / 8.0, e - 7", "(double)m / 16.0, e - 7"),
]

_FP8_MUTANT_RUNNER = _MUTANT_RUNNER.replace(
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs")',
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs", '
    '"oracle_decode_fp8_pairs", "oracle_e4m3_table")').replace(
    "T._pins_pass()", "T._fp8_pins_pass()")


@pytest.mark.parametrize("name,old,new", FP8_MUTANTS, ids=[m[0] for m in FP8_MUTANTS])
def test_fp8_pins_catch_planted_mistakes(name, old, new, tmp_path):
    import subprocess
    import sys

    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutant), "-lm"], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = _FP8_MUTANT_RUNNER.format(root=os.path.dirname(here), tests=here, so=str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode < 0 or "PINS_FAIL" in r.stdout, \
        f"no pin noticed the planted mistake: {name}\n{r.stdout}\n{r.stderr[-2000:]}"


def test_unmutated_oracle_passes_the_fp8_pins():
    assert _fp8_pins_pass()


# ---------------------------------------------------------------- x-packed layout
# "Paged Attention Kernel Architecture for BI-V100", section 3 (Paged K/V
# Gather): key cache [num_blocks, kv_heads, head_dim / x, block_size, x] with
# x = 16 / sizeof(element) (8 for bf16), value cache [num_blocks, kv_heads,
# head_dim, block_size].

def _xpacked_problem(seed=0, lens=(1, 15, 16, 17, 40, 33), H_q=8, H_kv=2, D=64, BS=16):
    spec = workloads.custom_spec("xp", len(lens), H_q, H_kv, D, BS, list(lens))
    w = workloads.make(spec, seed=seed, poison="nan")
    return w, workloads.to_xpacked(w)


def test_xpacked_repack_follows_the_stated_layout():
    """Element by element, written from the layout's definition (not from the
    repack): kx[b, g, d // 8, t, d % 8] = K[b, g, t, d] and vt[b, g, d, t] = V[b, g, t, d]."""
    w, x = _xpacked_problem(1, BS=32, D=128)
    k = w.k_cache.view(torch.int16)
    v = w.v_cache.view(torch.int16)
    kx = x.kx.view(torch.int16)
    vt = x.vt.view(torch.int16)
    assert tuple(kx.shape) == (k.shape[0], k.shape[1], k.shape[3] // 8, k.shape[2], 8)
    assert tuple(vt.shape) == (v.shape[0], v.shape[1], v.shape[3], v.shape[2])
    rng = np.random.default_rng(0)
    for _ in range(2000):
        b, g = int(rng.integers(k.shape[0])), int(rng.integers(k.shape[1]))
        t, d = int(rng.integers(k.shape[2])), int(rng.integers(k.shape[3]))
        assert kx[b, g, d // 8, t, d % 8] == k[b, g, t, d]
        assert vt[b, g, d, t] == v[b, g, t, d]


def test_xpacked_decode_equals_decode_of_the_same_values():
    """Same values in another order: the oracle's output is bit-identical."""
    for seed, BS, D in ((0, 16, 64), (1, 32, 128), (2, 16, 256)):
        w, x = _xpacked_problem(seed, BS=BS, D=D)
        assert np.array_equal(oracle.decode_xpacked(x), oracle.decode(w))


def test_xpacked_reads_only_the_sequences_rows():
    """NaN in every unread slot and block (the poison of the problem) never shows."""
    w, x = _xpacked_problem(3)
    assert np.isfinite(oracle.decode_xpacked(x)).all()


def _xpacked_pins_pass() -> bool:
    try:
        test_xpacked_decode_equals_decode_of_the_same_values()
        test_xpacked_reads_only_the_sequences_rows()
    except (AssertionError, oracle.OracleError, FloatingPointError):
        return False
    return True


XPACKED_MUTANTS = [
    ("slot and d/8 swapped",
     "((head * (size_t)(D / 8) + (size_t)(d / 8)) * c->BS + slot) * 8",
     "((head * (size_t)c->BS + slot) * (size_t)(D / 8) + (size_t)(d / 8)) * 8"),
    ("x = 16", "* c->BS + slot) * 8 +\n                                (size_t)(d % 8)",
     "* c->BS + slot) * 8 +\n                                (size_t)(d % 16)"),
    ("V token-major", "c->vt[(head * (size_t)D + (size_t)d) * c->BS + slot]",
     "c->vt[(head * (size_t)c->BS + slot) * D + (size_t)d]"),
    ("V of the K row", "return widen_bf16(c->vt[", "return widen_bf16(c->kx["),
]

_XPACKED_MUTANT_RUNNER = _MUTANT_RUNNER.replace(
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs")',
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs", '
    '"oracle_decode_xpacked_pairs")').replace("T._pins_pass()", "T._xpacked_pins_pass()")


@pytest.mark.parametrize("name,old,new", XPACKED_MUTANTS, ids=[m[0] for m in XPACKED_MUTANTS])
def test_xpacked_pins_catch_planted_mistakes(name, old, new, tmp_path):
    import subprocess
    import sys

    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutant), "-lm"], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = _XPACKED_MUTANT_RUNNER.format(root=os.path.dirname(here), tests=here, so=str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode < 0 or "PINS_FAIL" in r.stdout, \
        f"no pin noticed the planted mistake: {name}\n{r.stdout}\n{r.stderr[-2000:]}"


def test_unmutated_oracle_passes_the_xpacked_pins():
    assert _xpacked_pins_pass()


# ---------------------------------------------------------------- multi-token decode
# AstrAI CUDA Kernels page, "Q Scheduling and KV Addressing" (ragged qo_indptr)
# and "Python Wrappers" (is_causal): each sequence's last q_len tokens query the
# cache; with the causal mask query i sees the tokens t <= L - q_len + i.

def _multi_problem(seed, lens, qlens, H_q, H_kv, D, BS):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    K = [_bf16(torch.randn(L, H_kv, D, generator=g)) for L in lens]
    V = [_bf16(torch.randn(L, H_kv, D, generator=g)) for L in lens]
    kc, vc, bt, sl = _page(K, V, BS, rng)
    qo = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = _bf16(torch.randn(int(qo[-1]), H_q, D, generator=g))
    scale = float(np.float32(1.0 / math.sqrt(D)))
    return q, K, V, oracle.MultiInputs(q, kc, vc, bt, sl, scale), qo, scale


MULTI_CASES = [
    # seed, lens, qlens, H_q, H_kv, D, BS
    (1, [37, 100, 5], [1, 4, 5], 4, 2, 64, 16),
    (2, [16, 17, 33, 64], [2, 0, 7, 3], 8, 2, 32, 16),
    (3, [129, 8], [16, 8], 6, 1, 64, 32),
]


@pytest.mark.parametrize("seed,lens,qlens,H_q,H_kv,D,BS", MULTI_CASES)
def test_multi_matches_torch_sdpa_with_a_causal_mask(seed, lens, qlens, H_q, H_kv, D, BS):
    """torch float64 attention over the unpaged K/V with the mask written from
    the definition: query i of a sequence sees t <= L - q_len + i."""
    q, K, V, x, qo, scale = _multi_problem(seed, lens, qlens, H_q, H_kv, D, BS)
    got = oracle.decode_multi(x, qo, causal=True)
    for s, (L, ql) in enumerate(zip(lens, qlens)):
        if ql == 0:
            continue
        G = H_q // H_kv
        k = K[s].double().transpose(0, 1).repeat_interleave(G, dim=0)[None]  # [1, H_q, L, D]
        v = V[s].double().transpose(0, 1).repeat_interleave(G, dim=0)[None]
        qq = q[qo[s]:qo[s + 1]].double().transpose(0, 1)[None]              # [1, H_q, ql, D]
        mask = torch.tensor([[t <= L - ql + i for t in range(L)] for i in range(ql)])
        ref = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(got[qo[s]:qo[s + 1]], ref[0].transpose(0, 1).numpy(),
                                   rtol=0, atol=1e-12)


def test_multi_rows_equal_single_token_decodes_of_their_prefixes():
    """Row (s, i) is the single-token decode of sequence s cut at L - q_len + i + 1;
    without the mask, of the whole sequence."""
    q, K, V, x, qo, scale = _multi_problem(4, [40, 70], [3, 6], 8, 2, 64, 16)
    rows_s = np.repeat(np.arange(2), np.diff(qo))
    rows_i = np.arange(qo[-1]) - qo[rows_s]
    lens = x.lens[rows_s]
    for causal in (True, False):
        cut = lens - (np.diff(qo)[rows_s] - rows_i - 1) if causal else lens
        single = oracle.Inputs(q, x.k, x.v, x.bt[rows_s], cut.astype(np.int32), scale)
        assert np.array_equal(oracle.decode_multi(x, qo, causal=causal), oracle.decode(single))


def test_multi_with_one_query_per_sequence_is_the_decode():
    w = workloads.make("tiny", poison="nan")
    inp = oracle.Inputs.from_workload(w)
    qo = np.arange(inp.num_seqs + 1, dtype=np.int32)
    x = oracle.MultiInputs(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    assert np.array_equal(oracle.decode_multi(x, qo), oracle.decode(inp))


def test_multi_rejects_bad_offsets():
    q, K, V, x, qo, scale = _multi_problem(5, [10, 20], [2, 3], 4, 2, 32, 16)
    bad = qo.copy()
    bad[1] = 11  # q_len 11 > L = 10
    bad[2] = 14
    with pytest.raises((oracle.OracleError, ValueError)):
        oracle.decode_multi(oracle.MultiInputs(torch.zeros(14, 4, 32, dtype=torch.bfloat16),
                                               x.k, x.v, x.bt, x.lens, scale), bad)


def _multi_pins_pass() -> bool:
    try:
        for case in MULTI_CASES:
            test_multi_matches_torch_sdpa_with_a_causal_mask(*case)
        test_multi_rows_equal_single_token_decodes_of_their_prefixes()
    except (AssertionError, oracle.OracleError, FloatingPointError, ValueError):
        return False
    return True


MULTI_MUTANTS = [
    ("query sees one token too many", "const int seen = causal ? L - ql + i + 1 : L;",
     "const int seen = causal ? L - ql + i + 2 : L;"),
    ("query sees its own token not", "const int seen = causal ? L - ql + i + 1 : L;",
     "const int seen = causal ? L - ql + i : L;"),
    ("queries aligned to the start", "const int seen = causal ? L - ql + i + 1 : L;",
     "const int seen = causal ? i + 1 : L;"),
    ("query row of the first token", "const size_t r = (size_t)qo_indptr[s] + (size_t)i;",
     "const size_t r = (size_t)qo_indptr[s];"),
]

_MULTI_MUTANT_RUNNER = _MUTANT_RUNNER.replace(
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs")',
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs", "oracle_decode_multi")'
).replace("T._pins_pass()", "T._multi_pins_pass()")


@pytest.mark.parametrize("name,old,new", MULTI_MUTANTS, ids=[m[0] for m in MULTI_MUTANTS])
def test_multi_pins_catch_planted_mistakes(name, old, new, tmp_path):
    import subprocess
    import sys

    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutant), "-lm"], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = _MULTI_MUTANT_RUNNER.format(root=os.path.dirname(here), tests=here, so=str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode < 0 or "PINS_FAIL" in r.stdout, \
        f"no pin noticed the planted mistake: {name}\n{r.stdout}\n{r.stderr[-2000:]}"


def test_unmutated_oracle_passes_the_multi_pins():
    assert _multi_pins_pass()
