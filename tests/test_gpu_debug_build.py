"""The debug build: the same kernels compiled with SDPA_DEBUG, whose
device-side bounds checks guard the stores of O, LSE, dQ, dK and dV, the fp32
dQ accumulator's reductions and the shared-memory staging; a failed check
skips the access and sets SDPA_STATUS_BOUNDS instead of trapping.

The parity tests of every kernel family run in a child process with the
debug library loaded (SDPA_GB300_LIB) and must pass with the status word
clear. A debug flag then makes the forward's checks take O as one row shorter
than it is: the store of that row must be refused and reported, while the
buffer itself is full size, so nothing is ever written out of bounds."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from exact_attention_softmax_gb300 import build
    return build.build(debug=True)


def _child(debug_lib, args, timeout=1500):
    env = dict(os.environ, SDPA_GB300_LIB=debug_lib)
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def test_parity_tests_pass_under_the_debug_build(debug_lib):
    files = ["tests/test_gpu_fwd_tc.py", "tests/test_gpu_bwd_tc.py", "tests/test_gpu_blocksparse.py",
             "tests/test_gpu_masked.py", "tests/test_gpu_dropout.py", "tests/test_gpu_varlen_cross.py",
             "tests/test_gpu_strided.py", "tests/test_gpu_f32.py", "tests/test_gpu_persistent.py"]
    r = _child(debug_lib, ["-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                           "-k", "not dispatcher_shape", *files])
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


def test_refused_store_is_reported(debug_lib):
    code = textwrap.dedent("""
        import torch
        import exact_attention_softmax_gb300 as ops
        assert ops.sdpa_debug_build() == 1
        g = torch.Generator("cpu").manual_seed(5)
        for d in (64, 128):
            q, k, v = (torch.randn(1, 2, 200, d, generator=g).half().cuda() for _ in range(3))
            o = torch.full_like(q, float("nan"))
            lse = torch.full((1, 2, 200), float("nan"), device="cuda")
            ops.sdpa_debug_set(2)
            try:
                ops.sdpa_fwd(q, k, v, o, lse)
                try:
                    ops.sdpa_device_status()
                    raise AssertionError("the refused store was not reported")
                except ops.SdpaError as e:
                    assert e.code == -6, e
            finally:
                ops.sdpa_debug_set(0)
            # only the last row of O (unit 1, row 199) was refused
            assert torch.isnan(o[0, 1, 199]).all()
            assert not torch.isnan(o[0, 1, :199]).any() and not torch.isnan(o[0, 0]).any()
            ops.sdpa_fwd(q, k, v, o, lse)
            assert ops.sdpa_device_status() == 0 and not torch.isnan(o).any()
        print("ok")
    """)
    r = _child(debug_lib, ["-c", code], timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_normal_build_has_no_checks():
    import exact_attention_softmax_gb300 as ops
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    assert ops.sdpa_debug_build() == 0
