"""paged_attn_decode_static: decode for callers that cannot allocate device memory.

Some callers run inside a host framework that owns all device memory (a serving
engine that reserves the whole HBM for its KV-cache pool, a plugin host that
forbids allocation) or cannot afford cudaMalloc's implicit synchronisation in
the decode loop.  This entry point takes its scratch from a fixed 4 MiB array
compiled into the library instead of allocating.  The test calls it through the
C ABI and checks it against the allocating entry point, twice in a row (the
array keeps the previous call's contents, so the second call shows that what
must start at zero is cleared).  It lives in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
STATIC_SCRATCH_ERROR = -9


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_decode_gb300 import build

    build.build()
    import paged_kv_gqa_decode_gb300 as pa

    return pa.load()


def _c_call(lib, fn, w, out, stream):
    """Call a decode entry point of the C ABI with raw pointers."""
    num_seqs, H_q, D = w.q.shape
    _, H_kv, BS, _ = w.k_cache.shape
    return getattr(lib, fn)(
        ctypes.c_void_p(w.q.data_ptr()), ctypes.c_void_p(w.k_cache.data_ptr()),
        ctypes.c_void_p(w.v_cache.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(w.block_tables.data_ptr()), ctypes.c_void_p(w.seq_lens.data_ptr()),
        int(num_seqs), int(H_q), int(H_kv), int(D), int(w.block_tables.shape[1]), int(BS),
        ctypes.c_float(w.scale), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("name", ["tiny", "llama8b", "qwen100k", "ragged256", "gqa8"])
def test_static_scratch_matches_the_allocating_entry_point(lib, name):
    w = workloads.make(name, device="cuda", poison="nan")
    stream = torch.cuda.current_stream()
    ref = torch.empty_like(w.q)
    assert _c_call(lib, "paged_attn_decode", w, ref, stream) == 0
    torch.cuda.synchronize()
    want = ref.float().cpu().double().numpy()
    for _ in range(2):  # the array keeps the last call's contents between calls
        out = torch.full_like(w.q, float("nan"))
        assert _c_call(lib, "paged_attn_decode_static", w, out, stream) == 0
        torch.cuda.synchronize()
        got = out.float().cpu().double().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def test_static_scratch_rejects_sizes_beyond_its_limit(lib):
    # Find a supported shape whose split-KV state needs more than the 4 MiB array
    # on this device (on a 152-SM GB300: head_dim 128 with 16 query heads per KV
    # head), and check that the call is refused before anything is launched.
    shape = None
    for D in (128, 256, 64):
        for G in (16, 12, 8):
            need = lib.paged_attn_workspace_bytes(4, 2 * G, 2, D, 4, 16)
            if need > 4 << 20:
                shape = (D, G)
                break
        if shape:
            break
    if shape is None:
        pytest.skip("every supported shape fits in 4 MiB on this device")
    D, G = shape
    sp = workloads.custom_spec("too_big", 4, 2 * G, 2, D, 16, [64] * 4)
    w = workloads.make(sp, seed=3, device="cuda")
    out = torch.zeros_like(w.q)
    rc = _c_call(lib, "paged_attn_decode_static", w, out, torch.cuda.current_stream())
    assert rc == STATIC_SCRATCH_ERROR
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0  # nothing was launched
