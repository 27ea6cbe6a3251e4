"""More work items than SMs on the d <= 64 forward, whose CTAs are persistent:
each CTA claims (head, 256-row) items one after another and carries its
barrier phases, the deferred epilogue, the additive mask's slot counters and
the dropout counters from one item into the next. These batches have 240
items (2 x 40 heads x 3 items of 256, 256 and 88 rows) on at most 152 CTAs,
so that hand-over runs many times per CTA. Every (batch, head) unit is
compared with the fp64 oracle: O and LSE by max-abs error, each gradient by
its relative Frobenius error per unit. The backward runs on the same inputs. Plain bf16, the additive mask (per head and shared across the batch,
which also reorders the items, or one per (batch, head)) and dropout are
covered; the plain fp16 path has its many-item cases in the full-size
workload tests."""
import numpy as np
import pytest
import torch

import exact_attention_softmax_gb300 as ops
from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

B, H, L = 2, 40, 600
SEED = 0x243F6A8885A308D3


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _call(x, causal, scale, bwd, mask=None, dropout=None):
    """Forward (and backward) through the C ABI with canary-padded outputs."""
    from _gpu import check_guard, cuda, f64, guarded_empty
    dev = cuda()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lb, lse = guarded_empty(tuple(q.shape[:-1]), torch.float32, dev)
    m = None if mask is None else mask.to(dev)
    if m is not None:
        ops.sdpa_fwd_masked(q, k, v, m, o, lse, scale=scale, is_causal=causal)
    elif dropout is not None:
        ops.sdpa_fwd_dropout(q, k, v, dropout, SEED, o, lse, scale=scale, is_causal=causal)
    else:
        ops.sdpa_fwd(q, k, v, o, lse, scale=scale, is_causal=causal)
    out, bufs = [o, lse], [ob, lb]
    if bwd:
        do = x["do"].to(dev)
        gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
        g = [b[1] for b in gb]
        if m is not None:
            ops.sdpa_bwd_masked(q, k, v, o, lse, do, m, *g, scale=scale, is_causal=causal)
        elif dropout is not None:
            ops.sdpa_bwd_dropout(q, k, v, o, lse, do, dropout, SEED, *g, scale=scale, is_causal=causal)
        else:
            ops.sdpa_bwd(q, k, v, o, lse, do, *g, scale=scale, is_causal=causal)
        out += g
        bufs += [b[0] for b in gb]
    assert ops.sdpa_device_status() == 0
    for b in bufs:
        check_guard(b)
    return [f64(t) for t in out]


def _oracle(x, causal, scale, bwd, mask=None, dropout=None):
    from _gpu import f64
    from oracle import attn_bwd_ref, attn_fwd_ref
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    kw = {}
    if mask is not None:
        kw["attn_mask"] = mask.double().numpy()
    if dropout is not None:
        kw.update(dropout_p=dropout, dropout_seed=SEED)
    out = list(attn_fwd_ref(q, k, v, scale, causal, **kw))
    if bwd:
        out += list(attn_bwd_ref(q, k, v, f64(x["do"]), scale, causal, **kw))
    return out


def _compare_units(got, ref, dtype):
    """Each (batch, head) unit on its own: forward max-abs, gradients by
    relative Frobenius error; rows with no visible key (LSE = -inf) must be
    empty on both sides."""
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, rel_fro
    for b in range(B):
        for h in range(H):
            o, lse, ro, rl = got[0][b, h], got[1][b, h], ref[0][b, h], ref[1][b, h]
            empty = np.isneginf(rl)
            assert np.array_equal(np.isneginf(lse), empty), (b, h)
            assert np.max(np.abs(o - ro)) <= FWD_ATOL[dtype], (b, h, float(np.max(np.abs(o - ro))))
            ok = ~empty
            if ok.any():
                assert np.max(np.abs(lse[ok] - rl[ok])) <= LSE_ATOL[dtype], (b, h)
            for name, g, r in zip(("dQ", "dK", "dV"), got[2:], ref[2:]):
                e = rel_fro(g[b, h], r[b, h])
                assert e <= GRAD_RTOL[dtype], (name, b, h, e)


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_plain_bf16_many_items(d, causal):
    x = wl.dense_inputs(B, H, L, L, d, "bf16", "normal", seed=61, with_do=True)
    scale = d ** -0.5
    bwd = True
    _compare_units(_call(x, causal, scale, bwd), _oracle(x, causal, scale, bwd), "bf16")


@pytest.mark.parametrize("dtype,d", [("f16", 32), ("f16", 64), ("bf16", 64)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shared", [True, False], ids=["per-head-shared-over-batch", "per-unit"])
def test_masked_many_items(dtype, d, causal, shared):
    x = wl.dense_inputs(B, H, L, L, d, dtype, "normal", seed=62, with_do=True)
    lead = (1, H) if shared else (B, H)
    mask = wl.attn_mask(lead + (L, L), dtype, seed=63, empty_rows=(5, 300))[..., :L]
    scale = d ** -0.5
    bwd = True
    got = _call(x, causal, scale, bwd, mask=mask)
    ref = _oracle(x, causal, scale, bwd, mask=mask)
    _compare_units(got, ref, dtype)


@pytest.mark.parametrize("dtype,d", [("f16", 32), ("bf16", 32), ("f16", 64), ("bf16", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_dropout_many_items(dtype, d, causal):
    x = wl.dense_inputs(B, H, L, L, d, dtype, "normal", seed=64, with_do=True)
    scale = d ** -0.5
    bwd = True
    got = _call(x, causal, scale, bwd, dropout=0.3)
    ref = _oracle(x, causal, scale, bwd, dropout=0.3)
    _compare_units(got, ref, dtype)
