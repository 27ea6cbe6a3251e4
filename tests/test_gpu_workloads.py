"""The five measured workloads at their full sizes, in the launch configuration
the benchmark times, checked against the fp64 oracle on sampled (batch, head)
units and rows (the oracle computes each sampled unit or row on its own)."""
import math

import numpy as np
import pytest
import torch

import exact_attention_softmax_gb300 as ops
from exact_attention_softmax_gb300 import workloads as wl
from oracle import attn_bwd_unit, attn_fwd_rows, attn_fwd_unit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _run(w, x):
    from _gpu import FWD_ATOL  # noqa: F401
    dev = torch.device("cuda", 0)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    kw = {}
    if w.varlen:
        kw = dict(cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=x["max_seqlen"])
    o, lse = ops.sdpa_fwd(q, k, v, scale=w.scale, is_causal=w.causal, **kw)
    grads = None
    if w.bwd:
        grads = ops.sdpa_bwd(q, k, v, o, lse, x["do"].to(dev), scale=w.scale, is_causal=w.causal)
    assert ops.sdpa_device_status() == 0
    return o.cpu(), lse.cpu(), None if grads is None else [g.cpu() for g in grads]


def _np(t):
    return t.double().numpy()


@pytest.mark.parametrize("name", ["dense_f16_d32", "causal_f16_d64", "varlen_f16_d64"])
def test_workload_sampled_units(name):
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, rel_fro
    w = wl.WORKLOADS[name]
    x = wl.workload_inputs(w, seed=0)
    o, lse, grads = _run(w, x)
    rng = np.random.default_rng(1)
    if w.varlen:
        cu = x["cu_seqlens"].numpy()
        for s in list(rng.choice(w.nseq, 4, replace=False)) + [int(np.argmax(np.diff(cu)))]:
            a, b = cu[s], cu[s + 1]
            h = int(rng.integers(w.H))
            ro, rl = attn_fwd_unit(_np(x["q"][a:b, h]), _np(x["k"][a:b, h]), _np(x["v"][a:b, h]), w.scale, w.causal)
            assert np.max(np.abs(_np(o[a:b, h]) - ro)) <= FWD_ATOL[w.dtype]
            assert np.max(np.abs(_np(lse[h, a:b]) - rl)) <= LSE_ATOL[w.dtype]
        return
    units = [(0, 0), (w.B - 1, w.H - 1)] + [tuple(rng.integers([w.B, w.H])) for _ in range(4)]
    for b, h in units:
        q, k, v = (_np(x[n][b, h]) for n in ("q", "k", "v"))
        ro, rl = attn_fwd_unit(q, k, v, w.scale, w.causal)
        assert np.max(np.abs(_np(o[b, h]) - ro)) <= FWD_ATOL[w.dtype]
        assert np.max(np.abs(_np(lse[b, h]) - rl)) <= LSE_ATOL[w.dtype]
        if grads is not None:
            rg = attn_bwd_unit(q, k, v, _np(x["do"][b, h]), w.scale, w.causal)
            for g, r in zip(grads, rg):
                assert rel_fro(_np(g[b, h]), r) <= GRAD_RTOL[w.dtype]


def test_long_causal_bf16_sampled():
    """B=2, H=16, L=16384, d=128 causal bf16: forward rows sampled across the
    sequence in four units; one full unit's gradients against the oracle."""
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, rel_fro
    w = wl.WORKLOADS["long_causal_bf16_d128"]
    x = wl.workload_inputs(w, seed=0)
    o, lse, grads = _run(w, x)
    rows = np.array([0, 1, 127, 128, 4095, 8191, 8192, 12000, 16383])
    for b, h in [(0, 0), (0, 15), (1, 7), (1, 15)]:
        k, v = _np(x["k"][b, h]), _np(x["v"][b, h])
        ro, rl = attn_fwd_rows(_np(x["q"][b, h][rows]), k, v, rows, w.scale, True)
        assert np.max(np.abs(_np(o[b, h][rows]) - ro)) <= FWD_ATOL[w.dtype]
        assert np.max(np.abs(_np(lse[b, h][rows]) - rl)) <= LSE_ATOL[w.dtype]
    # invariants that hold at any size: dK sums to zero over keys, dV sums to sum(dO)
    for b, h in [(0, 3), (1, 12)]:
        dk = _np(grads[1][b, h])
        dv = _np(grads[2][b, h])
        do = _np(x["do"][b, h])
        assert np.max(np.abs(dk.sum(0))) <= 2e-2 * np.abs(dk).sum(0).max()
        np.testing.assert_allclose(dv.sum(0), do.sum(0), atol=0.05 * math.sqrt(w.Lq))
    b, h = 1, 9
    rg = attn_bwd_unit(_np(x["q"][b, h]), _np(x["k"][b, h]), _np(x["v"][b, h]), _np(x["do"][b, h]), w.scale, True)
    for g, r in zip(grads, rg):
        assert rel_fro(_np(g[b, h]), r) <= GRAD_RTOL[w.dtype]
