"""Parity of the tensor-core backward (fp16 / bf16, d in {32, 64, 128}) with the
fp64 oracle through the C ABI: dQ, dK, dV by relative Frobenius error, with
canaries around every gradient tensor; ragged tails and Lq != Lk included."""
import pytest
import torch

from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


SHAPES = [(1, 1, 1, 1), (1, 2, 127, 127), (1, 1, 128, 128), (2, 1, 129, 129),
          (1, 2, 300, 300), (1, 1, 200, 333), (1, 1, 333, 200)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dense_bwd(dtype, d, causal, shape):
    from _gpu import assert_fwd_close, assert_grads_close, oracle_bwd, oracle_fwd, run_fwd_bwd
    B, H, Lq, Lk = shape
    x = wl.dense_inputs(B, H, Lq, Lk, d, dtype, "normal", seed=7)
    scale = d ** -0.5
    o, lse, dq, dk, dv = run_fwd_bwd(x, causal, scale)
    assert_fwd_close((o, lse), oracle_fwd(x, causal, scale), dtype)
    assert_grads_close((dq, dk, dv), oracle_bwd(x, causal, scale), dtype)


def test_bwd_repeatable_within_tolerance():
    """dQ is accumulated with fp32 reductions whose order may vary; two runs agree
    to well inside the tolerance."""
    from _gpu import rel_fro, run_fwd_bwd
    x = wl.dense_inputs(1, 2, 640, 640, 64, "f16", "normal", seed=8)
    a = run_fwd_bwd(x, True, 0.125)
    b = run_fwd_bwd(x, True, 0.125)
    for u, v in zip(a, b):
        assert rel_fro(u, v) < 1e-3


def test_d32_dispatcher_shape_trains():
    """The SDPA tutorial's dispatcher example times a [32, 32, 1024, 32] fp16
    batch ("Explicit Dispatcher Control"); its backward at full size, one
    (batch, head) unit in four against the oracle (the others by the same
    kernel on the same schedule)."""
    from _gpu import GRAD_RTOL, f64, rel_fro
    from oracle import attn_bwd_unit
    import exact_attention_softmax_gb300 as ops
    B, H, L, d = 32, 32, 1024, 32
    x = wl.dense_inputs(B, H, L, L, d, "f16", "normal", seed=13)
    dev = torch.device("cuda", 0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = ops.sdpa_fwd(q, k, v)
    g = [t.cpu() for t in ops.sdpa_bwd(q, k, v, o, lse, do)]
    assert ops.sdpa_device_status() == 0
    for b, h in [(0, 0), (5, 17), (19, 30), (31, 31)]:
        ref = attn_bwd_unit(*(f64(x[n][b, h]) for n in ("q", "k", "v", "do")), d ** -0.5, False)
        for name, got, r in zip(("dQ", "dK", "dV"), g, ref):
            e = rel_fro(f64(got[b, h]), r)
            assert e <= GRAD_RTOL["f16"], (name, b, h, e)


LENGTHS = [1, 0, 130, 7, 256, 300, 129]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_bwd(dtype, d, causal):
    """Packed (variable-length) batches: rows of a tile that belong to the next
    sequence must neither contribute nor receive gradients."""
    from _gpu import (assert_fwd_close, assert_grads_close, oracle_bwd_packed, oracle_fwd,
                      run_fwd_bwd_packed)
    x = wl.varlen_inputs(LENGTHS, 3, d, dtype, "normal", seed=12)
    scale = d ** -0.5
    o, lse, dq, dk, dv = run_fwd_bwd_packed(x, causal, scale)
    assert_fwd_close((o, lse), oracle_fwd(x, causal, scale, packed=True), dtype)
    assert_grads_close((dq, dk, dv), oracle_bwd_packed(x, causal, scale), dtype)
