"""The kernel's bounded waits, made to run out on purpose.

Every wait in the decode kernel (a consumer waiting for a page, the producer
waiting for a free ring slot or draining its copies, a combiner waiting for the
other parts of a split to be published) gives up after a bounded number of
polls, reports status bit 2 and lets the launch finish.  These tests use a test
build of the library (``build.build_wait_test``: the bf16 head_dim-128 kernels
with waits of a few milliseconds and two hooks, never part of the product) in
which

* CTA 0 leaves one ring slot without its copy, so that page's wait runs out;
  every CTA still completes the split-counter protocol, so the next call on
  the same workspace is correct without any reset;
* every combiner waits for one more published part than exists, so its wait
  runs out; that call leaves split counters set, and the workspace is usable
  again after it is zero-filled (``paged_attn_reset_workspace`` for the
  library-owned one).

Nothing here faults, traps or hangs: a skipped copy is simply never issued,
and every wait that runs out returns."""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

TIMEOUT = 4


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_decode_gb300 import build
    import paged_kv_gqa_decode_gb300 as pa

    build.build()
    test_lib = pa.load(build.build_wait_test())
    test_lib.paged_attn_test_set_wait_faults.argtypes = [ctypes.c_int, ctypes.c_int]
    test_lib.paged_attn_test_set_wait_faults.restype = ctypes.c_int
    yield pa.load(), test_lib
    test_lib.paged_attn_test_set_wait_faults(-1, 0)


def _call_ws(lib, w, out, ws):
    num_seqs, H_q, D = w.q.shape
    _, H_kv, BS, _ = w.k_cache.shape
    return lib.paged_attn_decode_ws(
        w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(), out.data_ptr(),
        w.block_tables.data_ptr(), w.seq_lens.data_ptr(), int(num_seqs), int(H_q), int(H_kv),
        int(D), int(w.block_tables.shape[1]), int(BS), ctypes.c_float(w.scale), ws.data_ptr(),
        ws.numel(), torch.cuda.current_stream().cuda_stream)


def _call_owned(lib, w, out):
    num_seqs, H_q, D = w.q.shape
    _, H_kv, BS, _ = w.k_cache.shape
    return lib.paged_attn_decode(
        w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(), out.data_ptr(),
        w.block_tables.data_ptr(), w.seq_lens.data_ptr(), int(num_seqs), int(H_q), int(H_kv),
        int(D), int(w.block_tables.shape[1]), int(BS), ctypes.c_float(w.scale),
        torch.cuda.current_stream().cuda_stream)


def _status(ws):
    return int(ws[:4].view(torch.int32).item())


def _setup(libs, name="llama8b"):
    prod, test = libs
    w = workloads.make(name, seed=71, device="cuda", poison="nan")
    ref = torch.empty_like(w.q)
    assert _call_owned(prod, w, ref) == 0
    need = test.paged_attn_workspace_bytes(*(int(x) for x in (
        w.q.shape[0], w.q.shape[1], w.k_cache.shape[1], w.q.shape[2], w.block_tables.shape[1],
        w.k_cache.shape[2])))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    return prod, test, w, ref, ws


def test_wait_test_build_computes_what_the_library_does(libs):
    prod, test, w, ref, ws = _setup(libs)
    test.paged_attn_test_set_wait_faults(-1, 0)
    out = torch.full_like(w.q, float("nan"))
    assert _call_ws(test, w, out, ws) == 0
    torch.cuda.synchronize()
    assert _status(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("unit", [0, 2, 7])
def test_a_page_wait_that_runs_out_is_reported_and_the_workspace_stays_clean(libs, unit):
    prod, test, w, ref, ws = _setup(libs)
    test.paged_attn_test_set_wait_faults(unit, 0)
    out = torch.full_like(w.q, float("nan"))
    assert _call_ws(test, w, out, ws) == 0  # the launch itself is fine
    torch.cuda.synchronize()  # ... and it returns
    assert _status(ws) & TIMEOUT
    # the next call on the same workspace (status word cleared, counters untouched)
    test.paged_attn_test_set_wait_faults(-1, 0)
    ws[:4].zero_()
    out2 = torch.full_like(w.q, float("nan"))
    assert _call_ws(test, w, out2, ws) == 0
    torch.cuda.synchronize()
    assert _status(ws) == 0
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))


def test_a_combine_wait_that_runs_out_is_reported_and_a_reset_recovers(libs):
    prod, test, w, ref, ws = _setup(libs)
    test.paged_attn_test_set_wait_faults(-1, 1)
    out = torch.full_like(w.q, float("nan"))
    assert _call_ws(test, w, out, ws) == 0
    torch.cuda.synchronize()
    assert _status(ws) & TIMEOUT
    test.paged_attn_test_set_wait_faults(-1, 0)
    ws.zero_()  # split counters may be left set: zero-fill before the next use
    out2 = torch.full_like(w.q, float("nan"))
    assert _call_ws(test, w, out2, ws) == 0
    torch.cuda.synchronize()
    assert _status(ws) == 0
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))


def test_reset_workspace_recovers_the_library_owned_workspace(libs):
    prod, test, w, ref, _ = _setup(libs)
    out = torch.empty_like(w.q)
    assert _call_owned(test, w, out) == 0  # creates the test library's own workspace
    test.paged_attn_test_set_wait_faults(-1, 1)
    assert _call_owned(test, w, out) == 0
    test.paged_attn_test_set_wait_faults(-1, 0)
    assert test.paged_attn_reset_workspace(torch.cuda.current_stream().cuda_stream) == 0
    out2 = torch.full_like(w.q, float("nan"))
    assert _call_owned(test, w, out2) == 0
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))
