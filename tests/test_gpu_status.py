"""Failure detection without a GPU fault: every mbarrier wait in the
tensor-core kernels gives up after about a second. A debug flag makes the
forward's producer skip its Q load, so the first wait runs out; the kernel then
drains and returns, the host reads SDPA_ERR_TIMEOUT from the device status
word, and the context stays usable for the next, normal call."""
import time

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


def test_timeout_is_reported_and_context_survives():
    from _gpu import assert_fwd_close, oracle_fwd, run_fwd
    dev = torch.device("cuda", 0)
    x = wl.dense_inputs(1, 2, 200, 200, 64, "f16", "normal", seed=2, with_do=False)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    assert ops.sdpa_device_status() == 0
    old = ops.sdpa_debug_set(1)
    try:
        t0 = time.time()
        ops.sdpa_fwd(q, k, v, scale=0.125)
        with pytest.raises(ops.SdpaError) as e:
            ops.sdpa_device_status()
        waited = time.time() - t0
    finally:
        ops.sdpa_debug_set(old)
    assert e.value.code == -4          # SDPA_ERR_TIMEOUT
    assert waited < 30
    assert ops.sdpa_device_status() == 0   # the word was cleared
    # the context still works and gives correct results
    got = run_fwd(x, False, 0.125)
    assert_fwd_close(got, oracle_fwd(x, False, 0.125), "f16")


def test_packed_sequence_longer_than_bound_is_reported():
    dev = torch.device("cuda", 0)
    x = wl.varlen_inputs([100, 300], 1, 64, "f16", "normal", seed=1, with_do=False)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    ops.sdpa_fwd(q, k, v, cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=256)
    with pytest.raises(ops.SdpaError) as e:
        ops.sdpa_device_status()
    assert e.value.code == -1
    assert ops.sdpa_device_status() == 0
