"""Host-side tests of the backward entries (m3_scan_bwd, m3_scan_bwd_prep): workspace sizes and
argument checks that return before any launch, so they run without a GPU."""
import ctypes
import os

import pytest

from state_space_sequence_04_b300 import binding

BF16, F32 = 0, 1


@pytest.fixture(scope="module")
def lib():
    from state_space_sequence_04_b300 import build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.load()


@pytest.mark.parametrize("shape", [
    (1, 8, 2, 64, 128, 3),    # R = 3
    (1, 8, 2, 12, 16, 1),     # P / 4 = 3: not a power of two
    (1, 8, 2, 256, 16, 1),    # P > 128
    (1, 8, 2, 64, 7, 1),      # N odd
    (1, 8, 2, 64, 258, 1),    # N > 256
])
def test_workspace_zero_for_unsupported_shapes(lib, shape):
    assert binding.m3_scan_bwd_workspace_size(*shape, BF16) == 0
    assert binding.m3_scan_bwd_prep_workspace_size(*shape, BF16) == 0


def test_workspace_sizes_grow_with_the_problem(lib):
    """Checkpoints every 8 tokens (R <= 2) or 4 (R >= 4), pair-block partial sums: the sizes are
    256-byte multiples, grow with batch and tokens, and the pre-activation entry's exceed the plain one's
    by at least Delta, lambda and the normalised rows (and, where the forward takes the shape, y_pre)."""
    for R in (1, 2, 4, 8):
        a = binding.m3_scan_bwd_workspace_size(1, 64, 4, 64, 128, R, BF16)
        b = binding.m3_scan_bwd_workspace_size(2, 64, 4, 64, 128, R, BF16)
        c = binding.m3_scan_bwd_workspace_size(1, 128, 4, 64, 128, R, BF16)
        assert a > 0 and a % 256 == 0 and b > a and c > a
        bth = 1 * 64 * 4
        chunk = 8 if R <= 2 else 4
        assert a >= 4 * 4 * (64 // chunk) * 128 * 64          # the checkpoints alone
        p = binding.m3_scan_bwd_prep_workspace_size(1, 64, 4, 64, 128, R, BF16)
        extra = 2 * 4 * bth + 2 * 2 * bth * R * 128 + 2 * 4 * bth * R
        assert p >= a + extra
    # P = 64 bf16 is a forward shape (room for y_pre); P = 4 is not
    g = binding.m3_scan_bwd_prep_workspace_size(1, 64, 4, 64, 128, 1, BF16)
    assert g >= binding.m3_scan_bwd_workspace_size(1, 64, 4, 64, 128, 1, BF16) + 2 * 64 * 4 * 64
    assert binding.m3_scan_bwd_prep_workspace_size(1, 8, 2, 4, 4, 1, F32) > 0


def _fake(n=64):
    """A 16-byte-aligned host buffer standing in for device pointers the checks never dereference."""
    buf = (ctypes.c_float * (n + 4))()
    addr = ctypes.addressof(buf)
    return buf, addr + ((-addr) % 16)


def test_plain_entry_rejects_before_any_launch(lib):
    keep, p = _fake()
    ptrs = [p] * 17
    args = ptrs[:7] + [1] + ptrs[7:9] + ptrs[9:16]
    ok_sizes = [1, 8, 2, 64, 128, BF16]
    f = lib.m3_scan_bwd
    # R = 3: unsupported; misaligned A: invalid; no workspace: workspace error
    assert f(*(ptrs[:7] + [3] + ptrs[7:9] + ptrs[9:16]), *ok_sizes, p, 1 << 30, None) == binding.M3_ERR_UNSUPPORTED
    bad = list(args)
    bad[4] = p + 4
    assert f(*bad, *ok_sizes, p, 1 << 30, None) == binding.M3_ERR_INVALID_ARG
    assert f(*args, *ok_sizes, None, 0, None) == binding.M3_ERR_WORKSPACE
    assert f(*args, 1, 8, 2, 64, 128, 7, p, 1 << 30, None) == binding.M3_ERR_INVALID_ARG   # io dtype


def test_prep_entry_takes_bf16_normalisation_and_normalisation_with_gate(lib):
    """The B / C normalisation's backward accepts bf16 io and the gate: the calls pass every argument
    check and reach the launch, which an armed host-made launch failure turns into M3_ERR_CUDA before
    any CUDA call."""
    keep, p = _fake()
    params = binding.PrepParams(p, 1, 1e-5, None, None, None, None, None)
    gated = binding.PrepParams(p, 1, 1e-5, None, None, None, None, p)
    f = lib.m3_scan_bwd_prep
    args = [p] * 7 + [1] + [p] * 2 + [p] * 13

    ws = (p + 255) & ~255   # a 256-byte-aligned stand-in for the workspace (never dereferenced here)

    def call(io, prm):
        return f(*args, 1, 8, 2, 64, 128, io, ctypes.byref(prm), ws, 1 << 30, None)

    try:
        assert lib.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 3) == 0
        assert call(BF16, params) == binding.M3_ERR_CUDA
        assert call(F32, gated) == binding.M3_ERR_CUDA
        assert call(BF16, gated) == binding.M3_ERR_CUDA
        assert lib.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 0) == 0
    finally:
        lib.m3_test_inject(0, 0)
    bad_eps = binding.PrepParams(p, 1, -1.0, None, None, None, None, None)
    assert call(F32, bad_eps) == binding.M3_ERR_INVALID_ARG
