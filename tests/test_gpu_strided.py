"""Dense attention on strided tensors, through sdpa_fwd_strided /
sdpa_bwd_strided (the binding routes any non-contiguous dense tensor there).

The SDPA tutorial's module (section "Causal Self Attention") projects x to a
[B, L, 3E] buffer, splits it into q, k, v and views each as
[B, L, H, d].transpose(1, 2): [B, H, L, d] tensors whose rows are 3E elements
apart and whose heads are d apart. These tests pass exactly such views, with
no copy, and write O, dQ, dK, dV into the same kind of views of [B, L, E] and
[B, L, 3E] buffers, then compare with the fp64 oracle on the contiguous
values and with the contiguous calls, which must agree bit for bit (dQ,
whose fp32 partial sums are added in an order that may vary, within
rounding)."""
import numpy as np
import pytest
import torch

import exact_attention_softmax_gb300 as ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _module_views(B, L, H, d, dtype, seed):
    """q, k, v as the tutorial's module makes them: views of one [B, L, 3E]
    projection output; plus dO as a view of a [B, L, E] buffer."""
    from _gpu import cuda
    g = torch.Generator("cpu").manual_seed(seed)
    E = H * d
    td = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    qkv = torch.randn(B, L, 3 * E, generator=g).to(td).to(cuda())
    q, k, v = (t.view(B, L, H, d).transpose(1, 2) for t in qkv.split(E, dim=2))
    dy = torch.randn(B, L, E, generator=g).to(td).to(cuda())
    do = dy.view(B, L, H, d).transpose(1, 2)
    return q, k, v, do


def _out_views(B, L, H, d, like):
    """O in a [B, L, E] buffer, dQ/dK/dV in a [B, L, 3E] buffer (the layout
    of the projection's gradient), all as [B, H, L, d] views."""
    E = H * d
    y = torch.full((B, L, E), float("nan"), dtype=like.dtype, device=like.device)
    dqkv = torch.full((B, L, 3 * E), float("nan"), dtype=like.dtype, device=like.device)
    o = y.view(B, L, H, d).transpose(1, 2)
    dq, dk, dv = (t.view(B, L, H, d).transpose(1, 2) for t in dqkv.split(E, dim=2))
    return y, o, dqkv, dq, dk, dv


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("bf16", 64), ("bf16", 128), ("f32", 16)])
@pytest.mark.parametrize("causal", [False, True])
def test_module_layout_fwd_bwd_against_oracle(dtype, d, causal):
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, f64, rel_fro
    from oracle import attn_bwd_ref, attn_fwd_ref
    B, L, H = 2, 300, 512 // d if dtype != "f32" else 4
    q, k, v, do = _module_views(B, L, H, d, dtype, seed=81)
    assert not q.is_contiguous() and q.stride(2) == 3 * H * d
    y, o, dqkv, dq, dk, dv = _out_views(B, L, H, d, q)
    scale = d ** -0.5
    _, lse = ops.sdpa_fwd(q, k, v, o, scale=scale, is_causal=causal)
    ops.sdpa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale=scale, is_causal=causal)
    assert ops.sdpa_device_status() == 0
    assert not torch.isnan(y).any() and not torch.isnan(dqkv).any()   # every element written
    qn, kn, vn, don = (f64(t) for t in (q, k, v, do))
    ro, rl = attn_fwd_ref(qn, kn, vn, scale, causal)
    assert np.max(np.abs(f64(o) - ro)) <= FWD_ATOL[dtype]
    assert np.max(np.abs(f64(lse) - rl)) <= LSE_ATOL[dtype]
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), attn_bwd_ref(qn, kn, vn, don, scale, causal)):
        e = rel_fro(f64(g), r)
        assert e <= GRAD_RTOL[dtype], f"{name} {e:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_module_layout_many_items(causal):
    """More work items than SMs on strided views: 2 x 40 heads x 3 query items
    (256, 256 and 88 rows) in the forward and x 5 key blocks in the
    backward, whose d = 64 kernels are persistent, so each CTA carries its
    state from one item to the next. Every (batch, head) unit is compared with
    the fp64 oracle."""
    from _gpu import FWD_ATOL, GRAD_RTOL, LSE_ATOL, f64, rel_fro
    from oracle import attn_bwd_ref, attn_fwd_ref
    B, L, H, d = 2, 600, 40, 64
    q, k, v, do = _module_views(B, L, H, d, "f16", seed=84)
    y, o, dqkv, dq, dk, dv = _out_views(B, L, H, d, q)
    scale = d ** -0.5
    _, lse = ops.sdpa_fwd(q, k, v, o, scale=scale, is_causal=causal)
    ops.sdpa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale=scale, is_causal=causal)
    assert ops.sdpa_device_status() == 0
    assert not torch.isnan(y).any() and not torch.isnan(dqkv).any()
    qn, kn, vn, don = (f64(t) for t in (q, k, v, do))
    ro, rl = attn_fwd_ref(qn, kn, vn, scale, causal)
    rg = attn_bwd_ref(qn, kn, vn, don, scale, causal)
    got_o, got_l = f64(o), f64(lse)
    got_g = [f64(t) for t in (dq, dk, dv)]
    for b in range(B):
        for h in range(H):
            assert np.max(np.abs(got_o[b, h] - ro[b, h])) <= FWD_ATOL["f16"], (b, h)
            assert np.max(np.abs(got_l[b, h] - rl[b, h])) <= LSE_ATOL["f16"], (b, h)
            for name, g, r in zip(("dQ", "dK", "dV"), got_g, rg):
                e = rel_fro(g[b, h], r[b, h])
                assert e <= GRAD_RTOL["f16"], (name, b, h, e)


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("bf16", 128), ("f16", 32)])
def test_strided_equals_contiguous_bit_for_bit(dtype, d):
    """The strided calls run the same arithmetic as the contiguous ones."""
    B, L, H = 2, 257, 4
    q, k, v, do = _module_views(B, L, H, d, dtype, seed=82)
    y, o, dqkv, dq, dk, dv = _out_views(B, L, H, d, q)
    oc, lc = ops.sdpa_fwd(q.contiguous(), k.contiguous(), v.contiguous(), is_causal=True)
    _, ls = ops.sdpa_fwd(q, k, v, o, is_causal=True)
    assert torch.equal(o, oc) and torch.equal(ls, lc)
    gc = ops.sdpa_bwd(q.contiguous(), k.contiguous(), v.contiguous(), oc, lc, do.contiguous(), is_causal=True)
    ops.sdpa_bwd(q, k, v, o, ls, do, dq, dk, dv, is_causal=True)
    assert ops.sdpa_device_status() == 0
    # dQ goes through fp32 reductions whose order may vary: within rounding
    assert torch.equal(dk, gc[1]) and torch.equal(dv, gc[2])
    assert torch.allclose(dq.float(), gc[0].float(), rtol=1e-2, atol=1e-3)


def test_mixed_layouts_and_batch_stride_only():
    """Contiguous k with strided q / v, and a padded batch stride."""
    from _gpu import FWD_ATOL, cuda, f64
    from oracle import attn_fwd_ref
    B, H, L, d = 3, 2, 200, 64
    g = torch.Generator("cpu").manual_seed(83)
    big = torch.randn(B, H, L + 56, d, generator=g).half().to(cuda())
    q = big[:, :, :L]                                   # row stride d, head stride (L + 56) d
    k = torch.randn(B, H, L, d, generator=g).half().to(cuda())
    v = torch.randn(B, L, H, d, generator=g).half().to(cuda()).transpose(1, 2)
    o, lse = ops.sdpa_fwd(q, k, v, is_causal=False)
    assert ops.sdpa_device_status() == 0
    ro, _ = attn_fwd_ref(f64(q), f64(k), f64(v), d ** -0.5, False)
    assert np.max(np.abs(f64(o) - ro)) <= FWD_ATOL["f16"]


def test_strides_that_break_alignment_are_refused():
    from _gpu import cuda
    B, H, L, d = 1, 2, 64, 64
    base = torch.zeros(B, H, L, d + 4, dtype=torch.float16, device=cuda())
    q = base[..., :d]                                   # rows 68 elements apart: not a multiple of 8
    k = v = torch.zeros(B, H, L, d, dtype=torch.float16, device=cuda())
    with pytest.raises(ops.SdpaError, match="multiples of 8"):
        ops.sdpa_fwd(q, k, v)
