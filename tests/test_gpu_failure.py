"""Failure paths on the GPU, without a fault, a trap or a hang.

- The tensor-core prefill's bounded-wait failure path: m3_test_inject arms a
  test instantiation of the kernel whose consumer warps, at a given chunk, wait
  with a 50 us limit on an mbarrier that nothing completes.  Both warp groups
  then give up, drain the copies and MMAs still in flight (normal 2 s limits),
  free TMEM and write M3_ERR_TIMEOUT to the status word.  The test reads the
  word, then checks that the next (normal) call is correct against the oracle
  and leaves the word at M3_OK.
- A launch failure made on the host: the entry point returns M3_ERR_CUDA and
  launches nothing (its outputs keep their contents).
"""
import pytest
import torch

from state_space_sequence_04_b300 import binding, synth

from parity_util import TOL, KEYS, assert_close, need_gpu, oracle_sampled

pytestmark = pytest.mark.gpu

# 2 x 148 heads = 296 sequences fill the 148 SMs x 2 CTA slots: one segment per
# sequence, so every CTA walks all 10 chunks and gives up at chunk 4.
W = synth.Workload("timeout_b2_h148_T640_P64_N128_R1_Q64", 2, 148, 640, 64, 128, 1, 64, "bf16")
SAMPLES = [(0, 0), (1, 147), (0, 77)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    binding.m3_test_inject(0, 0)
    yield
    binding.m3_test_inject(0, 0)


def _status(ws):
    return int(ws[:4].view(torch.int32).item())


def _check(inp, y, fin, what):
    ref = oracle_sampled(inp, SAMPLES)
    for b, h in SAMPLES:
        yr, hr, _ = ref[(b, h)]
        assert_close(y[b:b + 1, :, h:h + 1], yr, TOL["bf16"], f"{what} y (b={b},h={h})")
        assert_close(fin[b:b + 1, h:h + 1], hr, TOL["bf16"], f"{what} final (b={b},h={h})")


def test_prefill_timeout_is_reported_and_the_next_call_is_correct():
    path, launches = binding.m3_scan_fwd_plan(W.batch, W.seqlen, W.heads, W.headdim, W.dstate, W.rank, W.chunk,
                                              binding.M3_DTYPE_BF16)
    assert (path, launches) == (1, 1)
    inp = synth.make_inputs(W, seed=11, device="cuda")
    args = [inp[k] for k in KEYS]
    ws = binding.alloc_workspace(inp["x"].shape, W.dstate, W.rank, W.chunk, torch.bfloat16, "cuda")
    y = torch.zeros_like(inp["x"])
    fin = torch.zeros((W.batch, W.heads, W.dstate, W.headdim), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()

    assert binding.m3_test_inject(binding.M3_TEST_PREFILL_TIMEOUT, 4) == -1
    assert binding.m3_scan_fwd(*args, W.rank, W.chunk, y, fin, ws) == binding.M3_OK
    torch.cuda.synchronize()
    assert _status(ws) == binding.M3_ERR_TIMEOUT
    # the chunks before the one given up on were written; the final state was not
    assert float(fin.abs().max()) == 0.0
    assert float(y[:, :4 * W.chunk].float().abs().max()) > 0.0

    # the injection was used up: the next call runs the normal kernel
    assert binding.m3_test_inject(binding.M3_TEST_PREFILL_TIMEOUT, 0) == -1
    binding.m3_test_inject(0, 0)
    assert binding.m3_scan_fwd(*args, W.rank, W.chunk, y, fin, ws) == binding.M3_OK
    torch.cuda.synchronize()
    assert _status(ws) == binding.M3_OK
    _check(inp, y, fin, "after a timeout")


def test_host_launch_failure_launches_nothing():
    inp = synth.make_inputs(W, seed=12, device="cuda", seqlen=128)
    args = [inp[k] for k in KEYS]
    ws = binding.alloc_workspace(inp["x"].shape, W.dstate, W.rank, W.chunk, torch.bfloat16, "cuda")
    y = torch.full_like(inp["x"], 7.0)
    fin = torch.full((W.batch, W.heads, W.dstate, W.headdim), 7.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert binding.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 1) == 0
    assert binding.m3_scan_fwd(*args, W.rank, W.chunk, y, fin, ws) == binding.M3_ERR_CUDA
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()) and bool((fin == 7.0).all())
    assert binding.m3_test_inject(binding.M3_TEST_LAUNCH_FAILURE, 0) == 0
    assert binding.m3_scan_fwd(*args, W.rank, W.chunk, y, fin, ws) == binding.M3_OK
    torch.cuda.synchronize()
    assert _status(ws) == binding.M3_OK
    ref = oracle_sampled(inp, SAMPLES[:2])
    for b, h in SAMPLES[:2]:
        yr, hr, _ = ref[(b, h)]
        assert_close(y[b:b + 1, :, h:h + 1], yr, TOL["bf16"], f"after a launch failure y (b={b},h={h})")
