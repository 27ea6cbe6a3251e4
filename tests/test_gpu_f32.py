"""Parity of the fp32 path (plain FFMA + expf kernels) with the fp64 oracle,
through the C ABI. Includes the tiny [2,3,8] workload against its stored
golden values."""
import json
import math
import os

import numpy as np
import pytest
import torch

from exact_attention_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built(built_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_tiny_workload_matches_golden():
    from _gpu import run_fwd_bwd, rel_fro
    gold = json.load(open(os.path.join(HERE, "golden", "tiny_f32.json")))
    w = wl.WORKLOADS["tiny_f32"]
    x = wl.workload_inputs(w, seed=gold["seed"])
    o, lse, dq, dk, dv = run_fwd_bwd(x, False, w.scale)
    g = {k: np.array(v) for k, v in gold["outputs"].items()}
    assert np.max(np.abs(o.reshape(-1) - g["o"])) <= 1e-5
    assert np.max(np.abs(lse.reshape(-1) - g["lse"])) <= 1e-5
    for a, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        assert rel_fro(a.reshape(-1), g[name]) <= 1e-5


@pytest.mark.parametrize("B,H,Lq,Lk,d,causal", [
    (1, 1, 1, 1, 8, False), (2, 3, 127, 129, 16, False), (2, 3, 127, 129, 16, True),
    (1, 2, 300, 300, 64, True), (1, 1, 5, 200, 128, False), (1, 1, 200, 5, 32, True),
    (1, 1, 130, 130, 7, True)])
def test_f32_dense_fwd_bwd(B, H, Lq, Lk, d, causal):
    from _gpu import assert_fwd_close, assert_grads_close, oracle_bwd, oracle_fwd, run_fwd_bwd
    x = wl.dense_inputs(B, H, Lq, Lk, d, "f32", "normal", seed=11)
    scale = 1 / math.sqrt(d)
    o, lse, dq, dk, dv = run_fwd_bwd(x, causal, scale)
    assert_fwd_close((o, lse), oracle_fwd(x, causal, scale), "f32")
    assert_grads_close((dq, dk, dv), oracle_bwd(x, causal, scale), "f32")


@pytest.mark.parametrize("causal", [False, True])
def test_f32_packed_fwd(causal):
    from _gpu import assert_fwd_close, oracle_fwd, run_fwd
    x = wl.varlen_inputs([1, 0, 130, 7, 256], 2, 16, "f32", "normal", seed=5)
    got = run_fwd(x, causal, 0.25, packed=True)
    assert_fwd_close(got, oracle_fwd(x, causal, 0.25, packed=True), "f32")


@pytest.mark.parametrize("causal", [False, True])
def test_f32_packed_fwd_bwd(causal):
    from _gpu import assert_fwd_close, assert_grads_close, oracle_bwd_packed, oracle_fwd, run_fwd_bwd_packed
    x = wl.varlen_inputs([1, 0, 130, 7, 256], 2, 16, "f32", "normal", seed=6)
    o, lse, dq, dk, dv = run_fwd_bwd_packed(x, causal, 0.25)
    assert_fwd_close((o, lse), oracle_fwd(x, causal, 0.25, packed=True), "f32")
    assert_grads_close((dq, dk, dv), oracle_bwd_packed(x, causal, 0.25), "f32")
