"""Parity of packed cross-attention (queries and keys on their own token axes,
sdpa_fwd_varlen / sdpa_bwd_varlen) with the fp64 oracle through the C ABI, and
of a [B, L, H, d] batch read through uniform offsets. The batches are the
tutorial's NestedTensor batches (SDPA tutorial page, section "NestedTensor and
Dense tensor support") with the key side indexed separately; lengths mix
ragged tails, a sequence with keys but no queries, single-key sequences and
more queries than keys (causal rows past the last key see every key)."""
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


LQ = [130, 0, 257, 7, 1, 300, 64]
LK = [200, 5, 64, 7, 129, 1, 383]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_cross_fwd_bwd(dtype, d, causal):
    from _gpu import assert_fwd_close, assert_grads_close, oracle_varlen_cross, run_varlen_cross
    x = wl.varlen_cross_inputs(LQ, LK, 3, d, dtype, "normal", seed=21)
    scale = d ** -0.5
    got = run_varlen_cross(x, causal, scale)
    ref = oracle_varlen_cross(x, causal, scale)
    assert_fwd_close(got[:2], ref[:2], dtype)
    assert_grads_close(got[2:], ref[2:], dtype)
    # keys of the sequence without queries get exactly zero gradient
    a, b = sum(LK[:1]), sum(LK[:2])
    assert np.all(got[3][a:b] == 0) and np.all(got[4][a:b] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_cross_fwd_d32(causal):
    from _gpu import assert_fwd_close, oracle_varlen_cross, run_varlen_cross
    x = wl.varlen_cross_inputs(LQ, LK, 2, 32, "f16", "normal", seed=22, with_do=False)
    got = run_varlen_cross(x, causal, 0.2, bwd=False)
    assert_fwd_close(got, oracle_varlen_cross(x, causal, 0.2, bwd=False), "f16")


@pytest.mark.parametrize("causal", [False, True])
def test_cross_f32(causal):
    from _gpu import assert_fwd_close, assert_grads_close, oracle_varlen_cross, run_varlen_cross
    lq, lk = [5, 0, 40, 1, 33], [9, 3, 17, 6, 1]
    x = wl.varlen_cross_inputs(lq, lk, 2, 48, "f32", "normal", seed=23)
    got = run_varlen_cross(x, causal, 0.3)
    ref = oracle_varlen_cross(x, causal, 0.3)
    assert_fwd_close(got[:2], ref[:2], "f32")
    assert_grads_close(got[2:], ref[2:], "f32")


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("bf16", 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_blhd_batch_through_uniform_offsets(dtype, d, causal):
    """A [B, L, H, d] batch is the packed case with offsets s * L: its results
    equal the dense oracle on the [B, H, L, d] transpose."""
    from _gpu import assert_fwd_close, assert_grads_close, cuda, f64, oracle_bwd, oracle_fwd
    B, Lq, Lk, H = 2, 192, 320, 3
    x = wl.dense_inputs(B, H, Lq, Lk, d, dtype, "normal", seed=24)
    dev = cuda()
    blhd = {n: x[n].transpose(1, 2).contiguous() for n in ("q", "k", "v", "do")}
    q, do = blhd["q"].view(B * Lq, H, d).to(dev), blhd["do"].view(B * Lq, H, d).to(dev)
    k, v = blhd["k"].view(B * Lk, H, d).to(dev), blhd["v"].view(B * Lk, H, d).to(dev)
    cq = torch.arange(B + 1, dtype=torch.int32, device=dev) * Lq
    ck = torch.arange(B + 1, dtype=torch.int32, device=dev) * Lk
    scale = d ** -0.5
    o, lse = ops.sdpa_fwd_varlen(q, k, v, cq, ck, Lq, Lk, scale=scale, is_causal=causal)
    dq, dk, dv = ops.sdpa_bwd_varlen(q, k, v, o, lse, do, cq, ck, Lq, Lk, scale=scale, is_causal=causal)
    assert ops.sdpa_device_status() == 0
    T = lambda t, L: f64(t).reshape(B, L, H, d).transpose(0, 2, 1, 3)
    lse_bhl = f64(lse).reshape(H, B, Lq).transpose(1, 0, 2)
    assert_fwd_close((T(o, Lq), lse_bhl), oracle_fwd(x, causal, scale), dtype)
    assert_grads_close((T(dq, Lq), T(dk, Lk), T(dv, Lk)), oracle_bwd(x, causal, scale), dtype)


def test_cross_with_shared_offsets_matches_self_attention_call():
    """sdpa_fwd_varlen with cu_seqlens_k == cu_seqlens_q gives bit-identical
    results to the self-attention sdpa_fwd / sdpa_bwd packed calls."""
    from _gpu import cuda
    lens = [130, 7, 256, 1]
    x = wl.varlen_inputs(lens, 2, 64, "f16", "normal", seed=25)
    dev = cuda()
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    cu, m = x["cu_seqlens"].to(dev), x["max_seqlen"]
    a = ops.sdpa_fwd(q, k, v, cu_seqlens=cu, max_seqlen=m, is_causal=True)
    b = ops.sdpa_fwd_varlen(q, k, v, cu, cu, m, m, is_causal=True)
    ga = ops.sdpa_bwd(q, k, v, a[0], a[1], do, cu_seqlens=cu, max_seqlen=m, is_causal=True)
    gb = ops.sdpa_bwd_varlen(q, k, v, b[0], b[1], do, cu, cu, m, m, is_causal=True)
    assert ops.sdpa_device_status() == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(ga[1], gb[1]) and torch.equal(ga[2], gb[2])
    # dQ goes through fp32 atomics whose order may vary between runs
    assert torch.allclose(ga[0].float(), gb[0].float(), atol=2e-3, rtol=0)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_cross_lengths_outside_bounds_are_reported(dtype):
    """A key length above max_seqlen_k, or queries with no keys, set the
    SEQLEN status bit in the forward and in the backward; the other sequences
    are still computed."""
    from _gpu import GRAD_RTOL, cuda, rel_fro
    from oracle import attn_bwd_unit
    dev = cuda()
    for lq, lk, mk in (([64, 40], [64, 300], 256), ([64, 40], [64, 0], 64)):
        x = wl.varlen_cross_inputs(lq, lk, 1, 64, dtype, "normal", seed=26, with_do=True)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        cq, ck = x["cu_seqlens_q"].to(dev), x["cu_seqlens_k"].to(dev)
        o, lse = ops.sdpa_fwd_varlen(q, k, v, cq, ck, max(lq), mk, is_causal=False)
        with pytest.raises(ops.SdpaError) as e:
            ops.sdpa_device_status()
        assert e.value.code == -1
        assert ops.sdpa_device_status() == 0
        from oracle import attn_fwd_unit
        ref, _ = attn_fwd_unit(x["q"][:64, 0].double().numpy(), x["k"][:64, 0].double().numpy(),
                               x["v"][:64, 0].double().numpy(), 0.125)
        tol = 4e-3 if dtype == "f16" else 1e-5
        assert np.max(np.abs(o[:64, 0].double().cpu().numpy() - ref)) < tol
        grads = ops.sdpa_bwd_varlen(q, k, v, o, lse, do, cq, ck, max(lq), mk, is_causal=False)
        with pytest.raises(ops.SdpaError) as e:
            ops.sdpa_device_status()
        assert e.value.code == -1
        assert ops.sdpa_device_status() == 0
        rg = attn_bwd_unit(*(x[n][:64, 0].double().numpy() for n in ("q", "k", "v", "do")), 0.125)
        for name, g, r in zip(("dQ", "dK", "dV"), grads, rg):
            err = rel_fro(g[:64, 0].double().cpu().numpy(), r)
            assert err <= GRAD_RTOL[dtype], f"{name} {err:.3e}"
