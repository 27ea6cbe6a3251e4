"""Parity of attention with dropout (sdpa_fwd_dropout / sdpa_bwd_dropout)
with the fp64 oracle through the C ABI: both sides draw the keep pattern from
Philox4x32-10 with the same seed (the generator implemented independently on
each side and pinned to its published known-answer vectors). The SDPA
tutorial's call takes dropout_p (section "Causal Self Attention")."""
import numpy as np
import pytest
import torch

import exact_attention_softmax_gb300 as ops
from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SEED = 0x9E3779B97F4A7C15


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _run(x, p, seed, causal, scale, bwd=True):
    from _gpu import check_guard, cuda, f64, guarded_empty
    dev = cuda()
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    ob, o = guarded_empty(tuple(q.shape), q.dtype, dev)
    lb, lse = guarded_empty(tuple(q.shape[:-1]), torch.float32, dev)
    ops.sdpa_fwd_dropout(q, k, v, p, seed, o, lse, scale=scale, is_causal=causal)
    out, bufs = [o, lse], [ob, lb]
    if bwd:
        do = x["do"].to(dev)
        gb = [guarded_empty(tuple(t.shape), t.dtype, dev) for t in (q, k, v)]
        ops.sdpa_bwd_dropout(q, k, v, o, lse, do, p, seed, gb[0][1], gb[1][1], gb[2][1], scale=scale,
                             is_causal=causal)
        out += [g for _, g in gb]
        bufs += [b for b, _ in gb]
    assert ops.sdpa_device_status() == 0
    for b in bufs:
        check_guard(b)
    return tuple(f64(t) for t in out)


def _oracle(x, p, seed, causal, scale, bwd=True):
    from _gpu import f64
    from oracle import attn_bwd_ref, attn_fwd_ref
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out = attn_fwd_ref(q, k, v, scale, causal, dropout_p=p, dropout_seed=seed)
    if bwd:
        out = out + attn_bwd_ref(q, k, v, f64(x["do"]), scale, causal, dropout_p=p, dropout_seed=seed)
    return out


SHAPES = [(1, 2, 300, 333), (2, 1, 256, 200)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dropout_fwd_bwd(dtype, d, causal, shape):
    from _gpu import assert_fwd_close, assert_grads_close
    B, H, Lq, Lk = shape
    x = wl.dense_inputs(B, H, Lq, Lk, d, dtype, "normal", seed=61)
    scale = d ** -0.5
    got = _run(x, 0.3, SEED, causal, scale)
    ref = _oracle(x, 0.3, SEED, causal, scale)
    assert_fwd_close(got[:2], ref[:2], dtype)
    assert_grads_close(got[2:], ref[2:], dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_d32_forward_and_f32(causal):
    from _gpu import assert_fwd_close, assert_grads_close
    x = wl.dense_inputs(2, 3, 260, 190, 32, "f16", "normal", seed=62, with_do=False)
    got = _run(x, 0.5, 12345, causal, 0.2, bwd=False)
    assert_fwd_close(got, _oracle(x, 0.5, 12345, causal, 0.2, bwd=False), "f16")
    x = wl.dense_inputs(1, 2, 70, 45, 16, "f32", "normal", seed=63)
    got = _run(x, 0.25, 777, causal, 0.3)
    ref = _oracle(x, 0.25, 777, causal, 0.3)
    assert_fwd_close(got[:2], ref[:2], "f32")
    assert_grads_close(got[2:], ref[2:], "f32")


def test_dropout_zero_seed_and_lse():
    """p = 0 is the plain call bit for bit; the same seed reproduces O, another
    seed changes it; LSE is the plain LSE whatever p is."""
    from _gpu import cuda
    dev = cuda()
    x = wl.dense_inputs(1, 2, 384, 384, 64, "f16", "normal", seed=64)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    plain = ops.sdpa_fwd(q, k, v)
    zero = ops.sdpa_fwd_dropout(q, k, v, 0.0, SEED)
    assert torch.equal(plain[0], zero[0]) and torch.equal(plain[1], zero[1])
    a = ops.sdpa_fwd_dropout(q, k, v, 0.4, SEED)
    b = ops.sdpa_fwd_dropout(q, k, v, 0.4, SEED)
    c = ops.sdpa_fwd_dropout(q, k, v, 0.4, SEED + 1)
    assert torch.equal(a[0], b[0])
    assert not torch.equal(a[0], c[0])
    assert torch.allclose(a[1], plain[1], atol=1e-5, rtol=0)
    with pytest.raises(ops.SdpaError):
        ops.sdpa_fwd_dropout(q, k, v, 1.0, SEED)
    assert ops.sdpa_device_status() == 0
