"""The seeded input generator: determinism, shapes, block tables and poison placement."""
import numpy as np
import pytest
import torch

import workloads


def test_same_seed_same_inputs():
    a = workloads.make("tiny")
    b = workloads.make("tiny")
    for x, y in [(a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache)]:
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.seq_lens, b.seq_lens)


def test_tiny_matches_its_description():
    w = workloads.make("tiny")
    assert w.lens_list == [37, 100]
    assert tuple(w.q.shape) == (2, 4, 64)
    assert tuple(w.k_cache.shape) == (16, 2, 16, 64)
    assert w.max_blocks_per_seq == 7
    assert w.scale == 0.125
    used = [int(b) for s, L in enumerate(w.lens_list)
            for b in w.block_tables[s, : -(-L // 16)].tolist()]
    assert len(set(used)) == len(used) == 3 + 7
    assert w.poison_block not in used
    # unused table entries point at the poison block
    assert (w.block_tables[0, 3:] == w.poison_block).all()


def test_poison_lands_only_on_unread_rows():
    w = workloads.make("tiny", poison="nan")
    BS = 16
    for s, L in enumerate(w.lens_list):
        for t in range(L):
            b = int(w.block_tables[s, t // BS])
            assert torch.isfinite(w.k_cache[b, :, t % BS].float()).all()
            assert torch.isfinite(w.v_cache[b, :, t % BS].float()).all()
        if L % BS:
            b = int(w.block_tables[s, L // BS])
            assert torch.isnan(w.k_cache[b, :, L % BS:].float()).all()
    assert torch.isnan(w.k_cache[w.poison_block].float()).all()


@pytest.mark.parametrize("name", ["llama8b", "qwen100k", "ragged256", "gqa8"])
def test_length_draws(name):
    sp = workloads.spec(name)
    rng = np.random.default_rng(workloads.SEEDS[name])
    lens = sp.lens(rng, sp.num_seqs)
    assert len(lens) == sp.num_seqs
    assert lens.min() >= 1 and lens.max() <= sp.max_len
    assert -(-int(lens.max()) // sp.block_size) <= sp.max_blocks_per_seq
    if name == "ragged256":
        assert lens.min() >= 16 and lens.max() <= 32768
        assert len(np.unique(lens)) > 100  # genuinely ragged


def test_custom_spec_lengths():
    sp = workloads.custom_spec("edge", 4, 8, 2, 64, 16, [0, 1, 16, 17])
    w = workloads.make(sp, seed=5)
    assert w.lens_list == [0, 1, 16, 17]
    assert w.max_blocks_per_seq == 2


def test_roofline_bytes_of_the_tiny_case():
    """The roofline numerator for the tiny case, worked by hand: 137 tokens x 2
    KV heads x (K + V) x 64 x 2 bytes = 70,144 B; q and out 2 x 4 heads x 64 x 2 B
    each = 2,048 B; ceil(37/16) + ceil(100/16) = 10 block-table entries = 40 B."""
    import bench

    sp = workloads.spec("tiny")
    w = workloads.make("tiny", device="cpu")
    b = bench.algorithmic_bytes(sp, w.lens_list)
    assert b == {"kv": 70144, "q_out": 2048, "block_table": 40, "total": 72232}
    # the per-(sequence, KV head) split the CPU baseline uses adds up to the same
    assert sum(bench.group_bytes(sp, L) for L in w.lens_list for _ in range(sp.H_kv)) == 72232
