"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
symbol include/paged_attn.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import paged_kv_gqa_decode_gb300 as pa
from paged_kv_gqa_decode_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return pa.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(paged_(?:attn|kv)_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(pa.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_library_exports_only_the_c_abi(lib):
    # Anything else exported -- a C++ helper, a template's static local (a GNU
    # "unique" symbol, shared by every library in the process) -- would let two
    # copies of the library loaded side by side interfere with each other.
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    allowed = set(declared_functions()) | {"_init", "_fini", "__bss_start", "_edata", "_end"}
    extra = []
    for line in out.splitlines():
        parts = line.split()
        if len(parts) >= 3 and parts[-1] not in allowed:
            extra.append(line)
    assert not extra, extra


def test_build_targets_sm103a_only():
    assert pbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    assert pa.paged_attn_status_string(0) == "ok"
    for code in range(-10, 0):
        assert pa.paged_attn_status_string(code) != "unknown status"
    assert lib.paged_attn_version() >= 100


def _call(lib, **kw):
    args = dict(q=16, k=16, v=16, out=16, bt=16, sl=16, num_seqs=2, H_q=8, H_kv=2, D=128,
                maxb=4, BS=16, scale=0.125, stream=None)
    args.update(kw)
    return lib.paged_attn_decode(args["q"], args["k"], args["v"], args["out"], args["bt"],
                                 args["sl"], args["num_seqs"], args["H_q"], args["H_kv"],
                                 args["D"], args["maxb"], args["BS"], args["scale"],
                                 args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(H_q=6, H_kv=4), -2),          # H_q not a multiple of H_kv
    (dict(H_q=34, H_kv=2), -2),         # G = 17 > 16
    (dict(H_kv=0), -2),
    (dict(D=96), -3),
    (dict(D=512), -3),
    (dict(BS=8), -4),
    (dict(BS=64), -4),
    (dict(num_seqs=-1), -5),
    (dict(maxb=0), -5),
    (dict(scale=float("nan")), -8),
    (dict(scale=float("inf")), -8),
    (dict(q=None), -1),                 # null pointer
    (dict(out=24), -1),                 # not 16-byte aligned
    (dict(bt=4), -1),
])
def test_bad_arguments_rejected_on_host(lib, kw, code):
    assert _call(lib, **kw) == code


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, num_seqs=0, q=None, k=None, v=None, out=None, bt=None, sl=None) == 0


def test_workspace_query_rejects_bad_sizes(lib):
    assert lib.paged_attn_workspace_bytes(4, 6, 4, 128, 8, 16) == 0
    assert lib.paged_attn_workspace_bytes(4, 8, 2, 80, 8, 16) == 0


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        pa.load(str(tmp_path / "nope.so"))


def test_launch_flags_are_checked_on_the_host(lib):
    """Only the early-prologue bit is known; a rejected call changes nothing."""
    assert lib.paged_attn_set_launch_flags(1) == 0
    assert lib.paged_attn_set_launch_flags(2) == -10
    assert lib.paged_attn_set_launch_flags(-1) == -10
    assert lib.paged_attn_set_launch_flags(0) == 0
    with pytest.raises(pa.PagedAttnError):
        pa.paged_attn_set_launch_flags(4)
