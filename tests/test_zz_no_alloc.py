"""m3_scan_fwd_noalloc: the prefill for callers that cannot allocate device memory.

Such callers (an application that owns every device allocation, a serving
loop that forbids allocation once running, a plugin host without an allocator
callback) cannot hand m3_scan_fwd a workspace; m3_scan_fwd_noalloc uses the
library's fixed scratch array instead.  These tests call it through the C ABI
several times in a row (so later calls see the scratch array as earlier calls
left it) and check each result against the float64 oracle and against
m3_scan_fwd on the same inputs, with the parity tolerances of the other GPU
tests; m3_device_status, which reads the scratch array's status word, must
stay M3_OK.  A timeout made with m3_test_inject must show up in
m3_device_status, and the call after it must be correct again.  The file is
named to be collected last.
"""
import pytest
import torch

from state_space_sequence_04_b300 import binding, synth

from parity_util import TOL, KEYS, assert_close, need_gpu, oracle_sampled, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024     # M3_NOALLOC_SCRATCH_BYTES in include/m3.h

# One problem per path: CUDA-core kernels (scratch holds the chunk states) and
# the tensor-core kernel (scratch holds its status word).
CASES = [
    # name, Bt, H, T, P, N, R, Q, io, seed
    ("cuda_core_fp32", 2, 4, 1000, 64, 64, 1, 64, "fp32", 1),
    ("tensor_core_bf16", 2, 4, 700, 64, 128, 1, 64, "bf16", 2),
    ("cuda_core_fp32_again", 1, 4, 333, 32, 128, 2, 32, "fp32", 3),
    ("tensor_core_bf16_again", 1, 8, 300, 64, 128, 1, 64, "bf16", 4),
]
SAMPLES = [(0, 0), (0, 3)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    binding.m3_test_inject(0, 0)
    yield
    binding.m3_test_inject(0, 0)


def _run_both(Bt, H, T, P, N, R, Q, io, seed):
    w = synth.Workload("noalloc", Bt, H, T, P, N, R, Q, io)
    inp = synth.make_inputs(w, seed=seed)
    d = to_dev(inp)
    args = [d[k] for k in KEYS]
    need = binding.m3_scan_fwd_workspace_size(Bt, T, H, P, N, R, Q, binding.io_code(d["x"].dtype))
    assert 0 < need <= SCRATCH_BYTES
    y_ref, fin_ref = binding.scan_fwd(*args, R, Q)
    y = torch.full_like(y_ref, float("nan"))
    fin = torch.full_like(fin_ref, float("nan"))
    st = binding.m3_scan_fwd_noalloc(*args, R, Q, y, fin)
    assert st == binding.M3_OK, binding.m3_status_string(st)
    torch.cuda.synchronize()
    return inp, y, fin, y_ref, fin_ref


def test_noalloc_matches_the_oracle_and_scan_fwd_on_consecutive_calls():
    for name, Bt, H, T, P, N, R, Q, io, seed in CASES:
        inp, y, fin, y_ref, fin_ref = _run_both(Bt, H, T, P, N, R, Q, io, seed)
        assert torch.isfinite(y.float()).all(), name
        ref = oracle_sampled(inp, SAMPLES)
        for b, h in SAMPLES:
            yr, hr, _ = ref[(b, h)]
            assert_close(y[b:b + 1, :, h:h + 1], yr, TOL[io], f"{name}: y vs oracle (b={b},h={h})")
            assert_close(fin[b:b + 1, h:h + 1], hr, TOL[io], f"{name}: final_state vs oracle (b={b},h={h})")
        assert_close(y, y_ref, TOL[io], f"{name}: y vs m3_scan_fwd")
        assert_close(fin, fin_ref, TOL[io], f"{name}: final_state vs m3_scan_fwd")
        assert binding.m3_device_status() == binding.M3_OK, name


def test_noalloc_timeout_is_reported_by_device_status():
    name, Bt, H, T, P, N, R, Q, io, seed = CASES[1]
    # 8 sequences: each is cut into one-chunk segments, so every CTA of the full pass gives up at its chunk 0
    binding.m3_test_inject(binding.M3_TEST_PREFILL_TIMEOUT, 0)
    w = synth.Workload("noalloc", Bt, H, T, P, N, R, Q, io)
    d = to_dev(synth.make_inputs(w, seed=seed))
    args = [d[k] for k in KEYS]
    y = torch.zeros_like(d["x"])
    fin = torch.zeros((Bt, H, N, P), dtype=torch.float32, device="cuda")
    assert binding.m3_scan_fwd_noalloc(*args, R, Q, y, fin) == binding.M3_OK
    assert binding.m3_device_status(clear=True) == binding.M3_ERR_TIMEOUT
    assert binding.m3_device_status() == binding.M3_OK
    # the next call is normal again
    inp, y, fin, y_ref, fin_ref = _run_both(Bt, H, T, P, N, R, Q, io, seed)
    assert binding.m3_device_status() == binding.M3_OK
    assert_close(y, y_ref, TOL[io], "after a timeout: y vs m3_scan_fwd")
    assert_close(fin, fin_ref, TOL[io], "after a timeout: final_state vs m3_scan_fwd")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # fp32, batch 4 x 64 heads x 4096 tokens needs ~0.5 GB of chunk states:
    # more than the fixed scratch, so the call must fail before any launch.
    lib = binding.load()
    need = binding.m3_scan_fwd_workspace_size(4, 4096, 64, 64, 128, 1, 64, binding.M3_DTYPE_F32)
    assert need > SCRATCH_BYTES
    p = [16 * (i + 1) for i in range(9)]   # aligned placeholders; never dereferenced
    st = lib.m3_scan_fwd_noalloc(p[0], p[1], p[2], p[3], p[4], p[5], p[6], 1, 64, p[7], p[8],
                                 4, 4096, 64, 64, 128, binding.M3_DTYPE_F32, None)
    assert st == binding.M3_ERR_WORKSPACE
    # invalid sizes keep m3_scan_fwd's own answer
    st = lib.m3_scan_fwd_noalloc(p[0], p[1], p[2], p[3], p[4], p[5], p[6], 3, 64, p[7], p[8],
                                 1, 128, 4, 64, 128, binding.M3_DTYPE_F32, None)
    assert st == binding.M3_ERR_UNSUPPORTED
