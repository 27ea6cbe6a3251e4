"""Parity of attention with an additive mask (sdpa_fwd_masked /
sdpa_bwd_masked) with the fp64 oracle through the C ABI. The SDPA tutorial's
module passes an attn_mask argument (section "Causal Self Attention"); the
masks here are seeded N(0,1) entries with about 10 % -inf, a query row
entirely -inf, padded row strides, per-head and broadcast masks."""
import numpy as np
import pytest
import torch

import exact_attention_softmax_gb300 as ops
from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _run(x, mask_full, lk, causal, scale, bwd=True):
    from _gpu import check_guard, cuda, f64, guarded_empty
    dev = cuda()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    m = mask_full.to(dev)[..., :lk]           # padded row stride kept on the device
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lb, lse = guarded_empty(tuple(q.shape[:-1]), torch.float32, dev)
    ops.sdpa_fwd_masked(q, k, v, m, o, lse, scale=scale, is_causal=causal)
    out, bufs = [o, lse], [ob, lb]
    if bwd:
        do = x["do"].to(dev)
        gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
        ops.sdpa_bwd_masked(q, k, v, o, lse, do, m, gb[0][1], gb[1][1], gb[2][1], scale=scale, is_causal=causal)
        out += [g for _, g in gb]
        bufs += [b for b, _ in gb]
    assert ops.sdpa_device_status() == 0
    for b in bufs:
        check_guard(b)
    return tuple(f64(t) for t in out)


def _oracle(x, mask_full, lk, causal, scale, bwd=True):
    from _gpu import f64
    from oracle import attn_bwd_ref, attn_fwd_ref
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    m = mask_full[..., :lk].double().numpy()
    out = attn_fwd_ref(q, k, v, scale, causal, attn_mask=m)
    if bwd:
        out = out + attn_bwd_ref(q, k, v, f64(x["do"]), scale, causal, attn_mask=m)
    return out


def _check_fwd(got, ref, dtype):
    from _gpu import assert_fwd_close
    o, lse = got
    ro, rlse = ref
    empty = np.isneginf(rlse)
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(o[empty] == 0)
    assert_fwd_close((o, np.where(empty, 0.0, lse)), (ro, np.where(empty, 0.0, rlse)), dtype)


SHAPES = [(1, 2, 300, 333), (2, 1, 256, 200), (1, 1, 129, 520)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_masked_fwd_bwd(dtype, d, causal, shape):
    from _gpu import assert_grads_close
    B, H, Lq, Lk = shape
    x = wl.dense_inputs(B, H, Lq, Lk, d, dtype, "normal", seed=51)
    mask = wl.attn_mask((B, H, Lq, Lk), dtype, seed=52, empty_rows=(3,))
    scale = d ** -0.5
    got = _run(x, mask, Lk, causal, scale)
    ref = _oracle(x, mask, Lk, causal, scale)
    _check_fwd(got[:2], ref[:2], dtype)
    assert_grads_close(got[2:], ref[2:], dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_masked_broadcast_and_d32_forward(causal):
    B, H, Lq, Lk, d = 2, 3, 260, 190, 32
    x = wl.dense_inputs(B, H, Lq, Lk, d, "f16", "normal", seed=53, with_do=False)
    mask = wl.attn_mask((Lq, Lk), "f16", seed=54)            # one mask for every (b, h)
    got = _run(x, mask, Lk, causal, 0.2, bwd=False)
    _check_fwd(got, _oracle(x, mask, Lk, causal, 0.2, bwd=False), "f16")


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("mshape", ["hqk", "qk", "b1qk"])
def test_masked_broadcast_bwd(d, mshape):
    """Masks shared across the batch ([H, Lq, Lk]), across everything
    ([Lq, Lk]) or across heads ([B, 1, Lq, Lk]) through the backward."""
    from _gpu import assert_grads_close
    B, H, Lq, Lk = 2, 3, 200, 260
    x = wl.dense_inputs(B, H, Lq, Lk, d, "bf16", "normal", seed=58)
    shape = {"hqk": (H, Lq, Lk), "qk": (Lq, Lk), "b1qk": (B, 1, Lq, Lk)}[mshape]
    mask = wl.attn_mask(shape, "bf16", seed=59, empty_rows=(5,))
    got = _run(x, mask, Lk, False, 0.125)
    ref = _oracle(x, mask, Lk, False, 0.125)
    _check_fwd(got[:2], ref[:2], "bf16")
    assert_grads_close(got[2:], ref[2:], "bf16")


@pytest.mark.parametrize("causal", [False, True])
def test_masked_f32(causal):
    from _gpu import assert_grads_close
    B, H, Lq, Lk, d = 1, 2, 70, 45, 16
    x = wl.dense_inputs(B, H, Lq, Lk, d, "f32", "normal", seed=55)
    mask = wl.attn_mask((H, Lq, Lk), "f32", seed=56, empty_rows=(0,), pad_to=1)
    got = _run(x, mask, Lk, causal, 0.3)
    ref = _oracle(x, mask, Lk, causal, 0.3)
    _check_fwd(got[:2], ref[:2], "f32")
    assert_grads_close(got[2:], ref[2:], "f32")


def test_triangular_mask_is_the_causal_call():
    """-inf above the diagonal through the mask equals is_causal = 1 within the
    fp16 tolerance (the two paths round S differently)."""
    from _gpu import cuda, f64
    dev = cuda()
    x = wl.dense_inputs(1, 2, 384, 384, 64, "f16", "normal", seed=57)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    tri = torch.zeros((384, 384), dtype=torch.float16, device=dev)
    tri.masked_fill_(torch.triu(torch.ones(384, 384, dtype=torch.bool, device=dev), 1), float("-inf"))
    a = ops.sdpa_fwd(q, k, v, is_causal=True)
    b = ops.sdpa_fwd_masked(q, k, v, tri)
    assert ops.sdpa_device_status() == 0
    assert np.max(np.abs(f64(a[0]) - f64(b[0]))) < 2e-3
    assert np.max(np.abs(f64(a[1]) - f64(b[1]))) < 1e-3
