"""Parity of the tensor-core forward (fp16 / bf16, d in {32, 64, 128}) with the
fp64 oracle through the C ABI: several 128-row tiles, ragged tails, Lq != Lk,
causal and non-causal, dense and packed, with canaries around every output."""
import pytest
import torch

from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


SHAPES = [(1, 1, 1, 1), (2, 2, 127, 127), (1, 2, 128, 128), (1, 1, 129, 129),
          (1, 2, 257, 257), (1, 1, 300, 520), (1, 1, 520, 300)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dense_fwd(dtype, d, causal, shape):
    from _gpu import assert_fwd_close, oracle_fwd, run_fwd
    B, H, Lq, Lk = shape
    x = wl.dense_inputs(B, H, Lq, Lk, d, dtype, "normal", seed=3, with_do=False)
    scale = d ** -0.5
    assert_fwd_close(run_fwd(x, causal, scale), oracle_fwd(x, causal, scale), dtype)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_fwd(dtype, d, causal):
    from _gpu import assert_fwd_close, oracle_fwd, run_fwd
    x = wl.varlen_inputs([1, 0, 130, 7, 256, 300], 2, d, dtype, "normal", seed=4, with_do=False)
    scale = d ** -0.5
    assert_fwd_close(run_fwd(x, causal, scale, packed=True), oracle_fwd(x, causal, scale, packed=True), dtype)


def test_uniform_inputs_d32():
    """torch.rand-style inputs (the dispatcher benchmark's distribution)."""
    from _gpu import assert_fwd_close, oracle_fwd, run_fwd
    x = wl.dense_inputs(2, 2, 384, 384, 32, "f16", "uniform", seed=9, with_do=False)
    scale = 32 ** -0.5
    assert_fwd_close(run_fwd(x, False, scale), oracle_fwd(x, False, scale), "f16")
