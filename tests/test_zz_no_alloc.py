"""The allocation-free backward, sdpa_bwd_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory when they run the
backward (a fixed-size memory pool, a plugin handed only its buffers, a host
that forbids cudaMalloc after start-up): the scratch comes from an array built
into the library. Its gradients must match those of sdpa_bwd with a
caller-provided workspace, on two calls in a row (the second call reuses the
array the first one left behind), and the fp64 oracle's; the second call must
leave the device's free memory unchanged. This file is collected last on
purpose.
"""
import ctypes

import pytest
import torch

from exact_attention_softmax_gb300 import _abi
from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    return _abi.load(built_lib)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,d,causal", [("f16", 64, True), ("bf16", 128, False), ("f32", 16, True)])
def test_noalloc_matches_workspace_backward_twice(lib, dtype, d, causal):
    from _gpu import GRAD_RTOL, f64, rel_fro
    B, H, L = 2, 3, 300
    code = {"f32": 0, "f16": 1, "bf16": 2}[dtype]
    dev = torch.device("cuda", 0)
    x = wl.dense_inputs(B, H, L, L, d, dtype, "normal", seed=21)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    _abi.check(lib.sdpa_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, L, L, d, scale, int(causal), None, code,
                            _stream()))
    # reference: the existing entry point with a caller-provided workspace
    ws = torch.empty(lib.sdpa_bwd_workspace_size(B, H, L, d, code), dtype=torch.uint8, device=dev)
    ref = [torch.empty_like(t) for t in (q, k, v)]
    _abi.check(lib.sdpa_bwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), *(_p(t) for t in ref),
                            B, H, L, L, d, scale, int(causal), None, code, _p(ws), ws.numel(), _stream()))
    from oracle import attn_bwd_ref
    exact = attn_bwd_ref(*(f64(x[n]) for n in ("q", "k", "v", "do")), scale, causal)
    outs = [[torch.full_like(t, float("nan")) for t in (q, k, v)] for _ in range(2)]
    torch.cuda.synchronize()
    for call, got in enumerate(outs):
        free_before = torch.cuda.mem_get_info(dev)[0]
        _abi.check(lib.sdpa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(do), *(_p(t) for t in got),
                                        B, H, L, L, d, scale, int(causal), code, _stream()))
        torch.cuda.synchronize()
        if call == 1:
            # the first call may load the scratch array; the second allocates nothing
            assert torch.cuda.mem_get_info(dev)[0] == free_before
        for name, g, r, ex in zip(("dQ", "dK", "dV"), got, ref, exact):
            e = rel_fro(f64(g), f64(r))
            assert e <= GRAD_RTOL[dtype], f"call {call}: {name} differs from sdpa_bwd by {e:.3e}"
            e = rel_fro(f64(g), ex)
            assert e <= GRAD_RTOL[dtype], f"call {call}: {name} differs from the oracle by {e:.3e}"


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    fake = ctypes.c_void_p(0x100000)
    B, H, L, d = 32, 8, 1024, 64   # needs about 65 MiB of scratch, above the 16 MiB built in
    rc = lib.sdpa_bwd_noalloc(*([fake] * 9), B, H, L, L, d, 0.125, 1, 1, None)
    assert rc == _abi.SDPA_ERR_WORKSPACE
    assert b"scratch" in lib.sdpa_last_error()
