"""The five measured workloads at their full sizes, in the launch configuration
the benchmark times, against the fp64 oracle. The dense fp16 batch (32 x 32 x
1024 x 32), the causal fp16 batch (32 x 8 x 1024 x 64, forward and backward)
and the 32-sequence packed batch are compared on EVERY (batch|sequence, head)
unit. The long causal bf16 batch (2 x 16 x 16384 x 128) is compared on four
whole (batch, head) slices of its forward, (0, 0), (0, 15), (1, 7) and
(1, 15), computed by the oracle a block of query rows at a time, and on one
whole unit of its backward, plus invariants of the backward that hold at any
size. Every output sits between canaries that catch stores outside it."""
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
    """Forward (and backward) of a workload through the C ABI, every output
    canary-padded. Returns CPU tensors."""
    from _gpu import check_guard, guarded_empty
    dev = torch.device("cuda", 0)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    kw = {}
    if w.varlen:
        kw = dict(cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=x["max_seqlen"])
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lshape = (w.H, q.shape[0]) if w.varlen else tuple(q.shape[:-1])
    lb, lse = guarded_empty(lshape, torch.float32, dev)
    ops.sdpa_fwd(q, k, v, o, lse, scale=w.scale, is_causal=w.causal, **kw)
    bufs = [ob, lb]
    grads = None
    if w.bwd:
        gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
        grads = ops.sdpa_bwd(q, k, v, o, lse, x["do"].to(dev), *[g for _, g in gb], scale=w.scale,
                             is_causal=w.causal, **kw)
        bufs += [b for b, _ in gb]
    assert ops.sdpa_device_status() == 0
    for b in bufs:
        check_guard(b)
    return o.cpu(), lse.cpu(), None if grads is None else [g.cpu() for g in grads]


def _np(t):
    return t.double().numpy()


@pytest.mark.parametrize("name", ["dense_f16_d32", "causal_f16_d64", "varlen_f16_d64"])
def test_workload_every_unit(name):
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, rel_fro
    w = wl.WORKLOADS[name]
    x = wl.workload_inputs(w, seed=0)
    o, lse, grads = _run(w, x)
    worst = [0.0, 0.0, 0.0]
    if w.varlen:
        cu = x["cu_seqlens"].numpy()
        for s in range(w.nseq):
            a, b = int(cu[s]), int(cu[s + 1])
            for h in range(w.H):
                ro, rl = attn_fwd_unit(_np(x["q"][a:b, h]), _np(x["k"][a:b, h]), _np(x["v"][a:b, h]), w.scale,
                                       w.causal)
                worst[0] = max(worst[0], float(np.max(np.abs(_np(o[a:b, h]) - ro))))
                worst[1] = max(worst[1], float(np.max(np.abs(_np(lse[h, a:b]) - rl))))
    else:
        for b in range(w.B):
            for h in range(w.H):
                q, k, v = (_np(x[n][b, h]) for n in ("q", "k", "v"))
                ro, rl = attn_fwd_unit(q, k, v, w.scale, w.causal)
                worst[0] = max(worst[0], float(np.max(np.abs(_np(o[b, h]) - ro))))
                worst[1] = max(worst[1], float(np.max(np.abs(_np(lse[b, h]) - rl))))
                if grads is not None:
                    rg = attn_bwd_unit(q, k, v, _np(x["do"][b, h]), w.scale, w.causal)
                    for g, r in zip(grads, rg):
                        worst[2] = max(worst[2], rel_fro(_np(g[b, h]), r))
    assert worst[0] <= FWD_ATOL[w.dtype], f"O max-abs {worst[0]:.3e}"
    assert worst[1] <= LSE_ATOL[w.dtype], f"LSE max-abs {worst[1]:.3e}"
    assert worst[2] <= GRAD_RTOL[w.dtype], f"worst per-unit gradient relative Frobenius {worst[2]:.3e}"


def test_long_causal_bf16_slices():
    """B=2, H=16, L=16384, d=128 causal bf16: four whole forward slices; one
    full unit's gradients; backward invariants on two more units."""
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, rel_fro
    w = wl.WORKLOADS["long_causal_bf16_d128"]
    x = wl.workload_inputs(w, seed=0)
    o, lse, grads = _run(w, x)
    chunk = 2048
    for b, h in [(0, 0), (0, 15), (1, 7), (1, 15)]:
        q, k, v = (_np(x[n][b, h]) for n in ("q", "k", "v"))
        for r0 in range(0, w.Lq, chunk):
            rows = np.arange(r0, min(r0 + chunk, w.Lq))
            kv = rows[-1] + 1           # causal: these rows see keys below kv only
            ro, rl = attn_fwd_rows(q[rows], k[:kv], v[:kv], rows, w.scale, True)
            err_o = float(np.max(np.abs(_np(o[b, h][r0:r0 + len(rows)]) - ro)))
            err_l = float(np.max(np.abs(_np(lse[b, h][r0:r0 + len(rows)]) - rl)))
            assert err_o <= FWD_ATOL[w.dtype], (b, h, r0, err_o)
            assert err_l <= LSE_ATOL[w.dtype], (b, h, r0, err_l)
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
