"""Host-side checks of the C ABI: the library builds for sm_103a, loads without
a GPU, exports every function include/sdpa.h declares, and rejects bad
arguments before anything reaches CUDA (no compute calls here)."""
import ctypes
import os
import re

import pytest

from exact_attention_softmax_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(0x100000)  # never dereferenced: every call below fails validation first


def _header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(sdpa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib(built_lib):
    return _abi.load(built_lib)


def test_library_exports_every_declared_function(lib):
    declared = _header_functions()
    assert {"sdpa_fwd", "sdpa_bwd", "sdpa_bwd_workspace_size", "sdpa_last_error"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(_abi.SIGNATURES) >= declared


def test_version_and_empty_error(lib):
    assert lib.sdpa_version() >= 100
    assert lib.sdpa_last_error() == b""


def _fwd(lib, B=1, H=1, Lq=4, Lk=4, d=64, scale=0.125, causal=0, cu=None, dtype=1, ptr=FAKE):
    return lib.sdpa_fwd(ptr, ptr, ptr, ptr, ptr, B, H, Lq, Lk, d, scale, causal, cu, dtype, None)


def test_argument_errors(lib):
    assert _fwd(lib, dtype=7) == _abi.SDPA_ERR_ARG
    assert b"dtype" in lib.sdpa_last_error()
    assert _fwd(lib, d=0) == _abi.SDPA_ERR_ARG
    assert _fwd(lib, B=-1) == _abi.SDPA_ERR_ARG
    assert _fwd(lib, scale=float("nan")) == _abi.SDPA_ERR_ARG
    assert _fwd(lib, scale=float("inf")) == _abi.SDPA_ERR_ARG
    assert _fwd(lib, causal=2) == _abi.SDPA_ERR_ARG
    assert _fwd(lib, Lk=0) == _abi.SDPA_ERR_ARG            # softmax over no keys
    assert _fwd(lib, ptr=ctypes.c_void_p(0)) == _abi.SDPA_ERR_ARG
    misaligned = ctypes.c_void_p(0x100008)
    assert _fwd(lib, ptr=misaligned) == _abi.SDPA_ERR_ARG   # TMA needs 16-byte aligned tensors


def test_unsupported_shapes(lib):
    assert _fwd(lib, d=48) == _abi.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, d=256, dtype=2) == _abi.SDPA_ERR_UNSUPPORTED
    assert _fwd(lib, d=129, dtype=0) == _abi.SDPA_ERR_UNSUPPORTED
    assert b"d" in lib.sdpa_last_error()


def test_empty_problems_are_noops(lib):
    # nothing to compute: returns OK without touching CUDA or the pointers
    assert _fwd(lib, Lq=0, ptr=ctypes.c_void_p(0)) == _abi.SDPA_OK
    assert _fwd(lib, B=0, ptr=ctypes.c_void_p(0)) == _abi.SDPA_OK
    assert _fwd(lib, H=0, ptr=ctypes.c_void_p(0)) == _abi.SDPA_OK


def test_workspace_size_and_errors(lib):
    assert lib.sdpa_bwd_workspace_size(0, 1, 1, 64, 1) == 0
    # fp32: only the row statistic D, rounded up to 256 bytes
    assert lib.sdpa_bwd_workspace_size(2, 1, 3, 8, 0) == 256
    # fp16: D plus an fp32 dQ accumulator
    B, H, L, d = 32, 8, 1024, 64
    n = B * H * L
    assert lib.sdpa_bwd_workspace_size(B, H, L, d, 1) == (n * 4 + 255) // 256 * 256 + n * d * 4
    args = [FAKE] * 9 + [B, H, L, L, d, 0.125, 1, None, 1]
    assert lib.sdpa_bwd(*args, FAKE, 16, None) == _abi.SDPA_ERR_WORKSPACE
    assert lib.sdpa_bwd(*args, None, 1 << 40, None) == _abi.SDPA_ERR_WORKSPACE
    assert b"workspace" in lib.sdpa_last_error()
    # packed: the workspace covers the Lq = total packed tokens (B = 1 in the size query)
    total = 700
    need_p = lib.sdpa_bwd_workspace_size(1, H, total, d, 1)
    args_p = [FAKE] * 9 + [5, H, total, 300, d, 0.125, 0, FAKE, 1]
    assert lib.sdpa_bwd(*args_p, FAKE, need_p - 1, None) == _abi.SDPA_ERR_WORKSPACE


def _fwd_varlen(lib, nseq=2, H=1, tq=8, tk=12, mq=5, mk=7, d=64, causal=0, cu_q=FAKE, cu_k=FAKE, dtype=1, ptr=FAKE):
    return lib.sdpa_fwd_varlen(ptr, ptr, ptr, ptr, ptr, nseq, H, tq, tk, mq, mk, d, 0.125, causal, cu_q, cu_k,
                               dtype, None)


def test_varlen_cross_argument_errors(lib):
    assert _fwd_varlen(lib, cu_k=None) == _abi.SDPA_ERR_ARG     # both offset arrays required
    assert b"offset" in lib.sdpa_last_error()
    assert _fwd_varlen(lib, cu_q=None) == _abi.SDPA_ERR_ARG
    assert _fwd_varlen(lib, mk=0) == _abi.SDPA_ERR_ARG          # queries but no keys anywhere
    assert _fwd_varlen(lib, tk=0) == _abi.SDPA_ERR_ARG
    assert _fwd_varlen(lib, tk=-1) == _abi.SDPA_ERR_ARG
    assert _fwd_varlen(lib, d=48) == _abi.SDPA_ERR_UNSUPPORTED
    assert _fwd_varlen(lib, ptr=ctypes.c_void_p(0x100008)) == _abi.SDPA_ERR_ARG
    # no query rows: a no-op that touches nothing
    assert _fwd_varlen(lib, tq=0, ptr=ctypes.c_void_p(0)) == _abi.SDPA_OK
    assert _fwd_varlen(lib, mq=0, ptr=ctypes.c_void_p(0)) == _abi.SDPA_OK
    assert _fwd_varlen(lib, nseq=0, ptr=ctypes.c_void_p(0)) == _abi.SDPA_OK
    # backward: the workspace covers the total query rows
    H, tq, d = 4, 700, 64
    need = lib.sdpa_bwd_workspace_size(1, H, tq, d, 1)
    args = [FAKE] * 9 + [3, H, tq, 900, 300, 400, d, 0.125, 1, FAKE, FAKE, 1]
    assert lib.sdpa_bwd_varlen(*args, FAKE, need - 1, None) == _abi.SDPA_ERR_WORKSPACE
    assert lib.sdpa_bwd_varlen(*(args[:19] + [None] + args[20:]), FAKE, need, None) == _abi.SDPA_ERR_ARG
    assert lib.sdpa_bwd_varlen(*(args[:15] + [48] + args[16:]), FAKE, need, None) == _abi.SDPA_ERR_UNSUPPORTED


def test_masked_and_blocksparse_argument_errors(lib):
    def fwdm(ptr=FAKE, mask=FAKE, sb=0, sh=0, sq=64, dtype=1, lk=60):
        return lib.sdpa_fwd_masked(ptr, ptr, ptr, ptr, ptr, 1, 1, 4, lk, 64, 0.125, 0, mask, sb, sh, sq, dtype, None)
    assert fwdm(mask=None) == _abi.SDPA_ERR_ARG
    assert fwdm(sq=59) == _abi.SDPA_ERR_ARG                # row stride below Lk
    assert fwdm(sq=60) == _abi.SDPA_ERR_ARG                # fp16: not a multiple of 8
    assert fwdm(sq=64, sb=4) == _abi.SDPA_ERR_ARG          # fp16: batch stride not a multiple of 8
    assert fwdm(mask=ctypes.c_void_p(0x100008)) == _abi.SDPA_ERR_ARG   # fp16: unaligned base
    assert fwdm(sh=-8) == _abi.SDPA_ERR_ARG
    assert b"mask" in lib.sdpa_last_error()

    def fwdb(mask=FAKE, sq=2, lk=256):
        return lib.sdpa_fwd_blocksparse(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, lk, 64, 0.125, 0, mask, 0, 0, sq, 1, None)
    assert fwdb(mask=None) == _abi.SDPA_ERR_ARG
    assert fwdb(sq=1) == _abi.SDPA_ERR_ARG                 # fewer than ceil(Lk / 128) key blocks per row
    args = [FAKE] * 9 + [1, 1, 200000, 256, 64, 0.125, 0, FAKE, 0, 0, 2, 1]
    need = lib.sdpa_bwd_workspace_size(1, 1, 200000, 64, 1)
    assert lib.sdpa_bwd_blocksparse(*args, FAKE, need, None) == _abi.SDPA_ERR_UNSUPPORTED   # Lq above 131072


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load(str(tmp_path / "nope.so"))


def test_python_binding_rejects_cpu_tensors(lib):
    """Every op takes CUDA tensors only: CPU tensors are refused with a clear
    error before any call reaches the library (there is no CPU implementation)."""
    import torch
    import exact_attention_softmax_gb300 as ops
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        ops.sdpa_fwd(q, q, q)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        ops.sdpa_fwd_dropout(q, q, q, 0.1, 7)
    lse = torch.zeros(1, 1, 8)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        ops.sdpa_bwd(q, q, q, q, lse, q)


def test_trace_events_argument_checks(lib):
    # setting and clearing the timing hook touches no CUDA state
    assert lib.sdpa_trace_events(2, None, None) == _abi.SDPA_ERR_ARG
    assert b"trace" in lib.sdpa_last_error()
    assert lib.sdpa_trace_events(0, FAKE, None) == _abi.SDPA_ERR_ARG
    assert lib.sdpa_trace_events(0, None, None) == _abi.SDPA_OK
    assert lib.sdpa_trace_events(1, None, None) == _abi.SDPA_OK


def test_strided_calls_check_their_strides(lib):
    st = (ctypes.c_longlong * 12)(*([8192, 2048, 64] * 4))
    ok = lib.sdpa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 32, 32, 64, 0.125, 0, None, 1, None)
    assert ok == _abi.SDPA_ERR_ARG and b"stride" in lib.sdpa_last_error()
    bad = (ctypes.c_longlong * 12)(*([8192, 2048, 68] * 4))        # rows 68 elements apart
    assert lib.sdpa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 32, 32, 64, 0.125, 0, bad, 1, None) == \
        _abi.SDPA_ERR_ARG
    assert b"multiples of 8" in lib.sdpa_last_error()
    neg = (ctypes.c_longlong * 12)(*([8192, -2048, 64] * 4))
    assert lib.sdpa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 32, 32, 64, 0.125, 0, neg, 1, None) == \
        _abi.SDPA_ERR_ARG
    # nothing to compute: returns OK before looking at the strides' values
    assert lib.sdpa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 0, 32, 64, 0.125, 0, st, 1, None) == _abi.SDPA_OK
