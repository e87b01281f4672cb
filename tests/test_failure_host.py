"""Failure injection on the host (no GPU needed): m3_test_inject's launch
failures.  An armed failure makes the next launching call return M3_ERR_CUDA
right after its argument checks, before any CUDA call, so the path runs here
without a device; calls that fail their checks, or have nothing to launch, do
not use one up."""
import os

import pytest

from state_space_sequence_04_b300 import binding

# 16-byte-aligned addresses standing in for device pointers: the checks never
# dereference them, and an armed failure returns before anything is launched.
P = [4096 * (i + 1) for i in range(16)]


@pytest.fixture(scope="module")
def lib():
    from state_space_sequence_04_b300 import build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.load()


@pytest.fixture(autouse=True)
def _disarm(lib):
    lib.m3_test_inject(0, 0)
    yield
    lib.m3_test_inject(0, 0)


def _scan(lib, ws_bytes, R=1, x=P[0]):
    # tensor-core sizes (bf16, N = 128, R = 1, chunk 64): the workspace is the status word only
    return lib.m3_scan_fwd(x, P[1], P[2], P[3], P[4], P[5], P[6], R, 64, P[7], None,
                           1, 128, 4, 64, 128, binding.M3_DTYPE_BF16, P[8], ws_bytes, None)


def test_armed_launch_failures_are_used_up_by_launching_calls(lib):
    need = binding.m3_scan_fwd_workspace_size(1, 128, 4, 64, 128, 1, 64, binding.M3_DTYPE_BF16)
    assert need > 0
    assert lib.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 3) == 0
    # rejected by the checks: nothing would launch, nothing is used up
    assert _scan(lib, need, x=None) == binding.M3_ERR_INVALID_ARG
    assert _scan(lib, need, R=3) == binding.M3_ERR_UNSUPPORTED
    assert _scan(lib, 0) == binding.M3_ERR_WORKSPACE
    # batch 0: nothing to launch
    st = lib.m3_decode_step(P[0], P[1], P[2], P[3], P[4], P[5], P[6], P[7], P[8], P[9],
                            0, 4, 64, 128, 1, binding.M3_DTYPE_BF16, None)
    assert st == binding.M3_OK
    assert lib.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 3) == 3
    # valid calls: each returns M3_ERR_CUDA and uses one up
    assert _scan(lib, need) == binding.M3_ERR_CUDA
    st = lib.m3_decode_step(P[0], P[1], P[2], P[3], P[4], P[5], P[6], P[7], P[8], P[9],
                            2, 4, 64, 128, 1, binding.M3_DTYPE_BF16, None)
    assert st == binding.M3_ERR_CUDA
    st = lib.m3_state_passing(P[0], P[1], P[2], None, None, 1, 2, 3, 16, 16, None)
    assert st == binding.M3_ERR_CUDA
    assert lib.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 0) == 0


def test_inject_arguments(lib):
    assert lib.m3_test_inject(7, 1) == binding.M3_ERR_INVALID_ARG
    assert lib.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, -1) == binding.M3_ERR_INVALID_ARG
    assert lib.m3_test_inject(binding.M3_TEST_PREFILL_TIMEOUT, 5) == -1
    assert lib.m3_test_inject(binding.M3_TEST_PREFILL_TIMEOUT, 2) == 5
    assert lib.m3_test_inject(0, 0) == 0
    assert lib.m3_test_inject(binding.M3_TEST_PREFILL_TIMEOUT, 1) == -1
