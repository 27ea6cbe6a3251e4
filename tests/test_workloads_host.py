"""The seeded input generators both sides of every parity test draw from,
and the algorithmic FLOP counts the benchmark divides by (no GPU)."""
import math

import pytest
import torch

from exact_attention_softmax_gb300 import workloads as wl


def test_dense_inputs_are_seeded_and_shaped():
    a = wl.dense_inputs(2, 3, 5, 7, 16, "bf16", "normal", seed=11)
    b = wl.dense_inputs(2, 3, 5, 7, 16, "bf16", "normal", seed=11)
    c = wl.dense_inputs(2, 3, 5, 7, 16, "bf16", "normal", seed=12)
    for n in ("q", "k", "v", "do"):
        assert torch.equal(a[n], b[n])
        assert not torch.equal(a[n], c[n])
        assert a[n].dtype == torch.bfloat16
    assert a["q"].shape == (2, 3, 5, 16) and a["do"].shape == (2, 3, 5, 16)
    assert a["k"].shape == (2, 3, 7, 16) and a["v"].shape == (2, 3, 7, 16)
    assert "do" not in wl.dense_inputs(1, 1, 4, 4, 8, "f16", "uniform", seed=1, with_do=False)
    u = wl.dense_inputs(1, 1, 64, 64, 32, "f32", "uniform", seed=3)["q"]
    assert float(u.min()) >= 0.0 and float(u.max()) < 1.0
    with pytest.raises(ValueError):
        wl.dense_inputs(1, 1, 4, 4, 8, "f16", "cauchy")


def test_varlen_lengths_and_offsets():
    lens = wl.varlen_lengths(32, 512, 0.5, seed=4)
    assert lens == wl.varlen_lengths(32, 512, 0.5, seed=4)
    assert len(lens) == 32 and all(1 <= n <= 512 for n in lens) and max(lens) == 512
    cu = wl.cu_seqlens_from(lens)
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and int(cu[-1]) == sum(lens)
    assert all(int(cu[i + 1]) - int(cu[i]) == lens[i] for i in range(len(lens)))
    x = wl.varlen_inputs(lens, 2, 8, "f16", seed=5)
    assert x["q"].shape == (sum(lens), 2, 8) and x["max_seqlen"] == 512 and x["lengths"] == lens


def test_varlen_cross_inputs():
    x = wl.varlen_cross_inputs([3, 5], [7, 2], 2, 8, "f16", seed=6)
    assert x["q"].shape == (8, 2, 8) and x["k"].shape == (9, 2, 8) and x["do"].shape == (8, 2, 8)
    assert x["cu_seqlens_q"].tolist() == [0, 3, 8] and x["cu_seqlens_k"].tolist() == [0, 7, 9]
    assert x["max_seqlen_q"] == 5 and x["max_seqlen_k"] == 7
    with pytest.raises(ValueError):
        wl.varlen_cross_inputs([3, 5], [7], 2, 8)


def test_block_mask():
    m = wl.block_mask((2, 64, 64), 0.5, seed=7, empty_rows=(3,))
    assert m.dtype == torch.uint8 and set(m.unique().tolist()) <= {0, 1}
    assert int(m[..., 3, :].sum()) == 0
    assert abs(float(m.float().mean()) - 0.5 * 63 / 64) < 0.03
    assert torch.equal(m, wl.block_mask((2, 64, 64), 0.5, seed=7, empty_rows=(3,)))


def test_attn_mask():
    m = wl.attn_mask((2, 50, 61), "f32", seed=8, neg_inf=0.1, empty_rows=(4,), pad_to=8)
    assert m.shape == (2, 50, 64) and m.dtype == torch.float32
    assert bool(torch.isneginf(m[:, 4, :]).all())
    rest = torch.cat([m[:, :4, :], m[:, 5:, :]], dim=1)
    frac = float(torch.isneginf(rest).float().mean())
    assert abs(frac - 0.1) < 0.02
    fin = rest[torch.isfinite(rest)]
    assert abs(float(fin.mean())) < 0.05 and abs(float(fin.std()) - 1.0) < 0.05
    assert wl.attn_mask((3, 9), "bf16", seed=9).dtype == torch.bfloat16


def test_flop_counts():
    w = wl.WORKLOADS["dense_f16_d32"]
    assert wl.fwd_flops(w) == 4.0 * w.B * w.H * w.Lq * w.Lk * w.d
    c = wl.WORKLOADS["causal_f16_d64"]
    assert wl.fwd_flops(c) == 2.0 * c.B * c.H * c.Lq * c.Lk * c.d
    assert wl.bwd_flops(c) == 2.5 * wl.fwd_flops(c)
    v = wl.WORKLOADS["varlen_f16_d64"]
    lens = [3, 5, 8]
    assert math.isclose(wl.fwd_flops(v, lens), 4.0 * v.H * v.d * (9 + 25 + 64))
