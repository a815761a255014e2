"""The Python binding's argument marshalling, on the CPU: every wrapper is called
with host tensors against a stand-in library that checks each call against the
argument types the binding declares for the real library (count and kind), and
that records the sizes passed.  No CUDA call is made."""
import ctypes

import pytest
import torch

import paged_kv_gqa_decode_gb300 as pa


class _Stream:
    cuda_stream = 0


class _Recorder:
    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        fn = getattr(self.real, name)

        def call(*args):
            types = fn.argtypes
            assert len(args) == len(types), (name, len(args), len(types))
            for a, t in zip(args, types):
                if t is ctypes.c_void_p:
                    assert a is None or isinstance(a, int), (name, a)
                elif t in (ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t):
                    assert isinstance(a, int), (name, a, t)
                elif t is ctypes.c_float:
                    assert isinstance(a, float), (name, a)
            self.calls.append((name, args))
            return 0

        return call


@pytest.fixture
def rec(monkeypatch):
    real = pa.load()  # the compiled library loads without a GPU
    r = _Recorder(real)
    monkeypatch.setattr(pa, "load", lambda path=None: r)
    return r


def _problem(num_seqs=3, H_q=8, H_kv=2, D=128, BS=16, nb=10, maxb=4):
    q = torch.zeros(num_seqs, H_q, D, dtype=torch.bfloat16)
    kc = torch.zeros(nb, H_kv, BS, D, dtype=torch.bfloat16)
    bt = torch.zeros(num_seqs, maxb, dtype=torch.int32)
    sl = torch.ones(num_seqs, dtype=torch.int32)
    return q, kc, kc.clone(), bt, sl


def test_every_wrapper_marshals_its_arguments(rec):
    s = _Stream()
    q, kc, vc, bt, sl = _problem()
    kn = torch.zeros(3, 2, 128, dtype=torch.bfloat16)
    pa.paged_attn_decode(q, kc, vc, bt, sl, 0.1, stream=s)
    pa.paged_attn_decode_static(q, kc, vc, bt, sl, 0.1, stream=s)
    pa.paged_attn_decode_checked(q, kc, vc, bt, sl, 0.1, torch.zeros(1, dtype=torch.int32),
                                 stream=s)
    pa.paged_attn_decode_ws(q, kc, vc, bt, sl, 0.1, torch.zeros(256, dtype=torch.uint8),
                            stream=s)
    pa.paged_kv_append(kn, kn, kc, vc, bt, sl, stream=s)
    pa.paged_attn_append_decode(q, kn, kn, kc, vc, bt, sl, 0.1, stream=s)
    # FP8 caches
    k8 = torch.zeros(10, 2, 16, 128, dtype=torch.uint8)
    ks = torch.ones(10, 2, 16, dtype=torch.float32)
    pa.paged_attn_decode_fp8(q, k8, k8, ks, ks, bt, sl, 0.1, stream=s)
    pa.paged_kv_append_fp8(kn, kn, k8, k8, ks, ks, bt, sl, stream=s)
    pa.paged_attn_append_decode_fp8(q, kn, kn, k8, k8, ks, ks, bt, sl, 0.1, stream=s)
    # x-packed caches
    kx = torch.zeros(10, 2, 16, 16, 8, dtype=torch.bfloat16)
    vt = torch.zeros(10, 2, 128, 16, dtype=torch.bfloat16)
    pa.paged_attn_decode_xpacked(q, kx, vt, bt, sl, 0.1, stream=s)
    # multi-token rows: 5 rows over 3 sequences
    qo = torch.tensor([0, 1, 3, 5], dtype=torch.int32)
    qm = torch.zeros(5, 8, 128, dtype=torch.bfloat16)
    km = torch.zeros(5, 2, 128, dtype=torch.bfloat16)
    pa.paged_attn_decode_multi(qm, kc, vc, qo, bt, sl, 0.1, 2, stream=s)
    pa.paged_attn_decode_multi(qm, kc, vc, qo, bt, sl, 0.1, 2, stream=s, causal=False)
    pa.paged_kv_append_multi(km, km, kc, vc, qo, bt, sl, stream=s)
    pa.paged_attn_append_decode_multi(qm, km, km, kc, vc, qo, bt, sl, 0.1, 2, stream=s,
                                      causal=False)
    pa.paged_attn_set_checks(10, torch.zeros(1, dtype=torch.int32))
    pa.paged_attn_set_checks(0, None)
    pa.paged_attn_set_launch_flags(pa.FLAG_EARLY_PROLOGUE)
    pa.paged_attn_set_launch_flags(0)
    pa.paged_attn_reset_workspace(stream=s)
    names = [n for n, _ in rec.calls]
    for n in ("paged_attn_decode", "paged_attn_decode_static", "paged_attn_decode_checked",
              "paged_attn_decode_ws", "paged_kv_append", "paged_attn_append_decode",
              "paged_attn_decode_fp8", "paged_kv_append_fp8", "paged_attn_append_decode_fp8",
              "paged_attn_decode_xpacked", "paged_attn_decode_multi_ex", "paged_kv_append_multi",
              "paged_attn_append_decode_multi", "paged_attn_set_checks",
              "paged_attn_set_launch_flags", "paged_attn_reset_workspace"):
        assert n in names, n
    calls = dict(rec.calls)
    # sizes: (num_seqs, H_q, H_kv, head_dim, max_blocks_per_seq, block_size) after the pointers
    assert calls["paged_attn_decode"][6:12] == (3, 8, 2, 128, 4, 16)
    assert calls["paged_attn_decode_fp8"][8:14] == (3, 8, 2, 128, 4, 16)
    assert calls["paged_kv_append_fp8"][8:13] == (3, 2, 128, 4, 16)
    assert calls["paged_attn_append_decode_fp8"][10:16] == (3, 8, 2, 128, 4, 16)
    # multi-token: (num_seqs, total_q, max_q_len, H_q, H_kv, head_dim, maxb, block_size)
    assert calls["paged_attn_append_decode_multi"][9:17] == (3, 5, 2, 8, 2, 128, 4, 16)
    assert calls["paged_attn_append_decode_multi"][18] == 0  # causal=False
    assert calls["paged_kv_append_multi"][7:13] == (3, 5, 2, 128, 4, 16)
    multi = [a for n, a in rec.calls if n == "paged_attn_decode_multi_ex"]
    assert [a[16] for a in multi] == [1, 0]


def test_wrappers_reject_mismatched_shapes(rec):
    s = _Stream()
    q, kc, vc, bt, sl = _problem()
    with pytest.raises(ValueError):
        pa.paged_kv_append(torch.zeros(3, 1, 128, dtype=torch.bfloat16),
                           torch.zeros(3, 1, 128, dtype=torch.bfloat16), kc, vc, bt, sl, stream=s)
    k8 = torch.zeros(10, 2, 16, 128, dtype=torch.uint8)
    with pytest.raises(ValueError):  # row floats of the wrong dtype
        pa.paged_kv_append_fp8(torch.zeros(3, 2, 128, dtype=torch.bfloat16),
                               torch.zeros(3, 2, 128, dtype=torch.bfloat16), k8, k8,
                               torch.ones(10, 2, 16, dtype=torch.float64),
                               torch.ones(10, 2, 16, dtype=torch.float64), bt, sl, stream=s)
    with pytest.raises(ValueError):  # qo_indptr of the wrong length
        pa.paged_attn_decode_multi(torch.zeros(5, 8, 128, dtype=torch.bfloat16), kc, vc,
                                   torch.tensor([0, 5], dtype=torch.int32), bt, sl, 0.1, 2,
                                   stream=s)
    assert rec.calls == []
