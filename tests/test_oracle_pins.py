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


# ---------------------------------------------------------------- FP8 cache write
# nvfp4-megamoe README, "FP8 KV Quantize/Dequant" and "Paged KV cache
# read/write".  Reading: a bf16 row x is stored as e4m3(x / f), f = max|x| / 448
# in float32 (1 for an all-zero row), rounding to the nearest e4m3 value with
# ties to the even code and saturation at 448.

def _finite_code_values():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    return codes, vals


def test_e4m3_encoding_matches_torch_float8_rounding():
    """The oracle's nearest-code search rounds as torch's float8_e4m3fn cast does
    (round to nearest even) on random values over the whole range, on every code
    value, on every midpoint between neighbouring codes (the ties) and just off
    each midpoint.  torch turns magnitudes past the tie at 464 into NaN where the
    reading saturates, so the comparison stops at 464."""
    rng = np.random.default_rng(0)
    parts = [rng.standard_normal(20000).astype(np.float32) * np.float32(2.0) ** e
             for e in range(-14, 9, 2)]
    _, vals = _finite_code_values()
    pos = np.unique(np.abs(vals))
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1].astype(np.float64) + pos[1:]) / 2)
    off = np.concatenate([np.nextafter(mids, np.float32(np.inf)),
                          np.nextafter(mids, np.float32(0))])
    x = np.concatenate(parts + [vals, mids, -mids, off, -off,
                                np.array([0.0, -0.0, 448.0, 460.0, 464.0], np.float32)])
    x = x[np.abs(x) <= 464]
    got = oracle.e4m3_encode(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]


def test_e4m3_encoding_saturates_and_round_trips_every_code():
    codes, vals = _finite_code_values()
    assert np.array_equal(oracle.e4m3_encode(vals), codes)  # every code is its own nearest
    big = np.array([465.0, 1e4, 3e38, np.inf], np.float32)
    assert np.array_equal(oracle.e4m3_encode(big), np.full(4, 0x7E, np.uint8))
    assert np.array_equal(oracle.e4m3_encode(-big), np.full(4, 0xFE, np.uint8))
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


def _bf16_rows(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)


def test_quantized_rows_decode_within_half_an_e4m3_step():
    """Decoding code x row float gives back x to within half an e4m3 step (2^-4
    relative in the normal range, 2^-10 of the row float below it); the largest
    magnitude of each row lands on +-448 exactly, and the float is that
    magnitude / 448 to within float32 rounding."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 128)).astype(np.float32) * \
        (np.float32(2.0) ** rng.integers(-20, 12, size=(64, 1))).astype(np.float32)
    xb = _bf16_rows(x)
    xd = xb.double().numpy()
    codes, f = oracle.quantize_rows_e4m3(xb)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * \
        f.astype(np.float64)[:, None]
    q = np.abs(xd) / f.astype(np.float64)[:, None]
    normal = q >= 2.0 ** -6
    err = np.abs(dec - xd)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xd[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(f[:, None], x.shape)[~normal])
    amax = np.abs(xd).max(axis=1)
    assert np.all(np.abs(f.astype(np.float64) * 448 - amax) <= amax * 2.0 ** -23)
    top = np.abs(xd).argmax(axis=1)
    assert np.all((codes[np.arange(64), top] & 0x7F) == 0x7E)


def test_rows_of_e4m3_values_quantize_exactly():
    """A row made of e4m3 values times 2^k with one element at +-448 * 2^k has row
    float 2^k and comes back code for code (the -0 code included)."""
    rng = np.random.default_rng(2)
    codes_all, _ = _finite_code_values()
    codes = rng.choice(codes_all, size=(40, 256)).astype(np.uint8)
    codes[np.arange(40), rng.integers(0, 256, 40)] = rng.choice([0x7E, 0xFE], 40)
    k = rng.integers(-12, 8, size=40)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double() * \
        torch.from_numpy(np.ldexp(1.0, k))[:, None]
    xb = vals.to(torch.bfloat16)
    assert torch.equal(xb.double(), vals)
    got, f = oracle.quantize_rows_e4m3(xb)
    assert np.array_equal(f, np.ldexp(1.0, k).astype(np.float32))
    assert np.array_equal(got, codes)


def test_all_zero_row_has_float_one():
    got, f = oracle.quantize_rows_e4m3(torch.zeros(3, 128, dtype=torch.bfloat16))
    assert np.array_equal(f, np.ones(3, np.float32)) and not got.any()


def _fp8_write_pins_pass() -> bool:
    try:
        test_e4m3_encoding_matches_torch_float8_rounding()
        test_e4m3_encoding_saturates_and_round_trips_every_code()
        test_quantized_rows_decode_within_half_an_e4m3_step()
        test_rows_of_e4m3_values_quantize_exactly()
        test_all_zero_row_has_float_one()
    except (AssertionError, oracle.OracleError, FloatingPointError, ValueError):
        return False
    return True


FP8_WRITE_MUTANTS = [
    ("ties to the odd code", "(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    ("rounds toward zero", "const double err = fabs(e4m3_value((uint8_t)c) - a);",
     "const double err = e4m3_value((uint8_t)c) <= a ? a - e4m3_value((uint8_t)c) : INFINITY;"),
    ("row float from 240", "amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 240.0f : 1.0f"),
    ("zero row float 0", "amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 448.0f : 0.0f"),
    ("multiplies by the float", "e4m3_encode((float)widen_bf16(x[d]) / f)",
     "e4m3_encode((float)widen_bf16(x[d]) * f)"),
    ("sign dropped", "return (uint8_t)(sign | best);", "return (uint8_t)best;"),
    ("amax of the signed values", "const float a = fabsf((float)widen_bf16(x[d]));",
     "const float a = (float)widen_bf16(x[d]);"),
]

_FP8_WRITE_MUTANT_RUNNER = _MUTANT_RUNNER.replace(
    '("oracle_decode", "oracle_decode_pairs", "oracle_partial_pairs")',
    '("oracle_e4m3_encode", "oracle_quantize_rows_e4m3")').replace(
    "T._pins_pass()", "T._fp8_write_pins_pass()")


@pytest.mark.parametrize("name,old,new", FP8_WRITE_MUTANTS, ids=[m[0] for m in FP8_WRITE_MUTANTS])
def test_fp8_write_pins_catch_planted_mistakes(name, old, new, tmp_path):
    import subprocess
    import sys

    src = open(oracle._SRC).read()
    assert src.count(old) == 1, name
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutant), "-lm"], check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = _FP8_WRITE_MUTANT_RUNNER.format(root=os.path.dirname(here), tests=here, so=str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode < 0 or "PINS_FAIL" in r.stdout, \
        f"no pin noticed the planted mistake: {name}\n{r.stdout}\n{r.stderr[-2000:]}"


def test_unmutated_oracle_passes_the_fp8_write_pins():
    assert _fp8_write_pins_pass()


def _fp8_exact_cache(seed, lens, H_kv=2, D=128, BS=16):
    """An FP8 problem whose every cache row is e4m3 codes x 2^k with one element at
    +-448 x 2^k (so quantizing its decoded values gives the row back exactly)."""
    spec = workloads.custom_spec("fp8exact", len(lens), 4 * H_kv, H_kv, D, BS, list(lens))
    w = workloads.make(spec, seed=seed, poison="none")
    rng = np.random.default_rng(seed)
    shape = tuple(w.k_cache.shape)
    codes_all, _ = _finite_code_values()
    codes = rng.choice(codes_all, size=(2,) + shape).astype(np.uint8)
    flat = codes.reshape(-1, D)
    flat[np.arange(flat.shape[0]), rng.integers(0, D, flat.shape[0])] = 0x7E
    scales = np.ldexp(1.0, rng.integers(-6, 4, size=(2,) + shape[:3])).astype(np.float32)
    f8 = oracle.Fp8Inputs(w.q, codes[0], codes[1], scales[0], scales[1], w.block_tables,
                          w.seq_lens, w.scale)
    return w, f8


def _newest_fp8_rows(f8):
    """Each sequence's newest K and V rows as bf16 values, read through the un-paged view."""
    vals = []
    for c8, sc in ((f8.k8, f8.ks), (f8.v8, f8.vs)):
        dec = torch.from_numpy(c8).view(torch.float8_e4m3fn).double() * \
            torch.from_numpy(sc).double().unsqueeze(-1)
        rows = torch.zeros(f8.num_seqs, f8.H_kv, f8.D, dtype=torch.float64)
        for s in range(f8.num_seqs):
            L = int(f8.lens[s])
            if L:
                pages = [int(f8.bt[s, i]) for i in range(-(-L // f8.BS))]
                flat = torch.cat([dec[b] for b in pages], dim=1)  # [H_kv, pages*BS, D]
                rows[s] = flat[:, L - 1]
        vals.append(rows.to(torch.bfloat16))
    return vals


def _fp8_append_round_trip(append_fp8):
    """Take each newest row out of an exact FP8 cache, poison its bytes and float,
    append its values back: bytes and floats come back bit for bit, nothing else moves."""
    _, f8 = _fp8_exact_cache(3, [1, 15, 16, 17, 40, 0, 33])
    k_new, v_new = _newest_fp8_rows(f8)
    hole = copy_fp8(f8)
    for s in range(hole.num_seqs):
        L = int(hole.lens[s])
        if L:
            b = int(hole.bt[s, (L - 1) // hole.BS])
            hole.k8[b, :, (L - 1) % hole.BS] = 0x7F
            hole.v8[b, :, (L - 1) % hole.BS] = 0x7F
            hole.ks[b, :, (L - 1) % hole.BS] = np.nan
            hole.vs[b, :, (L - 1) % hole.BS] = np.nan
    back = append_fp8(hole, k_new, v_new)
    assert np.array_equal(back.k8, f8.k8) and np.array_equal(back.v8, f8.v8)
    assert np.array_equal(back.ks, f8.ks) and np.array_equal(back.vs, f8.vs)


def copy_fp8(f8):
    import copy as _copy

    c = _copy.copy(f8)
    c.k8, c.v8, c.ks, c.vs = f8.k8.copy(), f8.v8.copy(), f8.ks.copy(), f8.vs.copy()
    return c


def _fp8_append_pins_pass(append_fp8) -> bool:
    try:
        _fp8_append_round_trip(append_fp8)
    except (AssertionError, oracle.OracleError, IndexError, ValueError):
        return False
    return True


def test_fp8_append_round_trip_restores_bytes_and_floats():
    _fp8_append_round_trip(oracle.append_fp8)


FP8_APPEND_MUTANTS = [
    ("slot from L", "out.k8[b, :, t % inp.BS, :] = kc[s]", "out.k8[b, :, L % inp.BS, :] = kc[s]"),
    ("float of V from K", "out.vs[b, :, t % inp.BS] = vf[s]", "out.vs[b, :, t % inp.BS] = kf[s]"),
    ("page of the next token", "b = int(inp.bt[s, t // inp.BS])", "b = int(inp.bt[s, L // inp.BS])"),
]


@pytest.mark.parametrize("name,old,new", FP8_APPEND_MUTANTS, ids=[m[0] for m in FP8_APPEND_MUTANTS])
def test_fp8_append_pins_catch_planted_mistakes(name, old, new):
    import inspect

    src = inspect.getsource(oracle.append_fp8)
    assert src.count(old) == 1, name
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    assert not _fp8_append_pins_pass(ns["append_fp8"]), f"no pin noticed: {name}"


# ---------------------------------------------------------------- multi-token append

MULTI_APPEND_LENS = [1, 15, 16, 17, 40, 0, 33, 5]
MULTI_APPEND_QLENS = [1, 3, 16, 2, 17, 0, 8, 7]


def _multi_append_problem(seed=12):
    spec = workloads.custom_spec("mapp", len(MULTI_APPEND_LENS), 8, 2, 64, 16, MULTI_APPEND_LENS)
    w = workloads.make(spec, seed=seed, poison="nan")
    qo = np.concatenate([[0], np.cumsum(MULTI_APPEND_QLENS)]).astype(np.int32)
    return oracle.Inputs.from_workload(w), qo


def _newest_rows(inp, qo):
    """Each sequence's last q_len cached rows (fewer when L < q_len: those rows stay
    zero), [total_q, H_kv, D], read through the un-paged view."""
    k = np.zeros((int(qo[-1]), inp.H_kv, inp.D), dtype=np.uint16)
    v = np.zeros_like(k)
    for s in range(inp.num_seqs):
        L, ql = int(inp.lens[s]), int(qo[s + 1] - qo[s])
        if L == 0:
            continue
        pages = [inp.bt[s, i] for i in range(-(-L // inp.BS))]
        fk = np.concatenate([inp.k[b] for b in pages], axis=1)
        fv = np.concatenate([inp.v[b] for b in pages], axis=1)
        for i in range(ql):
            t = L - ql + i
            if t >= 0:
                k[qo[s] + i], v[qo[s] + i] = fk[:, t], fv[:, t]
    return k, v


def _multi_append_pins(append_multi):
    inp, qo = _multi_append_problem()
    # one new token each: the single-token append
    ones = np.arange(inp.num_seqs + 1, dtype=np.int32)
    rng = np.random.default_rng(4)
    kn = rng.integers(0x4700, 0x4780, size=(inp.num_seqs, inp.H_kv, inp.D), dtype=np.uint16)
    vn = rng.integers(0xC700, 0xC780, size=kn.shape, dtype=np.uint16)
    a, b = append_multi(inp, ones, kn, vn), oracle.append(inp, kn, vn)
    assert np.array_equal(a.k, b.k) and np.array_equal(a.v, b.v)
    # round trip: the newest q_len rows taken out, poisoned and appended back
    k_new, v_new = _newest_rows(inp, qo)
    hole = oracle.Inputs.from_workload(workloads.make(workloads.custom_spec(
        "mapp", len(MULTI_APPEND_LENS), 8, 2, 64, 16, MULTI_APPEND_LENS), seed=12, poison="nan"))
    hole.k, hole.v = hole.k.copy(), hole.v.copy()
    for s in range(hole.num_seqs):
        L, ql = int(hole.lens[s]), int(qo[s + 1] - qo[s])
        for t in range(max(0, L - ql), L):
            bb = int(hole.bt[s, t // hole.BS])
            hole.k[bb, :, t % hole.BS] = 0x7FC0
            hole.v[bb, :, t % hole.BS] = 0x7FC0
    back = append_multi(hole, qo, k_new, v_new)
    assert np.array_equal(back.k, inp.k) and np.array_equal(back.v, inp.v)
    # exactly min(q_len, L) rows per sequence change
    big_k = rng.integers(0x4700, 0x4780, size=k_new.shape, dtype=np.uint16)
    big_v = rng.integers(0xC700, 0xC780, size=k_new.shape, dtype=np.uint16)
    out = append_multi(inp, qo, big_k, big_v)
    rows = sum(min(L, q) for L, q in zip(MULTI_APPEND_LENS, MULTI_APPEND_QLENS))
    assert int((out.k != inp.k).sum()) == rows * inp.H_kv * inp.D
    assert int((out.v != inp.v).sum()) == rows * inp.H_kv * inp.D
    got_k, _ = _newest_rows(out, qo)
    for s in range(inp.num_seqs):
        L, ql = int(inp.lens[s]), int(qo[s + 1] - qo[s])
        for i in range(ql):
            if L - ql + i >= 0:
                assert np.array_equal(got_k[qo[s] + i], big_k[qo[s] + i])


def _multi_append_pins_pass(append_multi) -> bool:
    try:
        _multi_append_pins(append_multi)
    except (AssertionError, oracle.OracleError, IndexError, ValueError):
        return False
    return True


def test_multi_append_is_the_append_for_one_token_and_round_trips():
    _multi_append_pins(oracle.append_multi)


MULTI_APPEND_MUTANTS = [
    ("one token later", "t = L - ql + i\n", "t = L - ql + i + 1\n"),
    ("row of the sequence index", "r = int(qo[s]) + i", "r = s + i"),
    ("negative tokens written", "if t < 0:\n                continue", "if t < -99:\n                continue"),
    ("v from k", "out.v[b, :, t % inp.BS, :] = vn[r]", "out.v[b, :, t % inp.BS, :] = kn[r]"),
]


@pytest.mark.parametrize("name,old,new", MULTI_APPEND_MUTANTS,
                         ids=[m[0] for m in MULTI_APPEND_MUTANTS])
def test_multi_append_pins_catch_planted_mistakes(name, old, new):
    import inspect

    src = inspect.getsource(oracle.append_multi)
    assert src.count(old) == 1, name
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)
    assert not _multi_append_pins_pass(ns["append_multi"]), f"no pin noticed: {name}"


def test_noncausal_multi_matches_torch_sdpa_without_a_mask():
    """Without the causal mask every query row of a sequence attends all its tokens:
    torch float64 SDPA over the un-paged K/V, no mask."""
    lens, qlens, H_q, H_kv, D, BS = [5, 40, 17], [2, 7, 17], 6, 2, 32, 16
    q, K, V, kc, vc, bt, sl = _random_problem(21, lens, H_q, H_kv, D, BS)
    g = torch.Generator().manual_seed(22)
    qm = _bf16(torch.randn(sum(qlens), H_q, D, generator=g))
    qo = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    x = oracle.MultiInputs(qm, kc, vc, bt, sl, 0.125)
    got = oracle.decode_multi(x, qo, causal=False)
    for s in range(len(lens)):
        rows = qm[qo[s]:qo[s + 1]]
        want = _sdpa(rows, [K[s]] * len(rows), [V[s]] * len(rows), 0.125)
        assert np.allclose(got[qo[s]:qo[s + 1]], want, rtol=0, atol=1e-12)
