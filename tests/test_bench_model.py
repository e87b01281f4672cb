"""The backward's cost model in bench.py against the figures derived by hand: 26 + 10R FLOPs per state
element and token (one forward evaluation plus the adjoint), and the bytes of every input read once and
every fp32 gradient written once."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_model", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_backward_flops_and_bytes_of_the_siso_workload():
    bench = _bench()
    from state_space_sequence_04_b300 import synth
    w = synth.SISO_1P5B
    th = w.batch * w.seqlen * w.heads                      # 1,048,576 (token, head) pairs
    assert bench.bwd_flops(w) == 36 * 128 * 64 * th        # 3.09e11
    # bf16 x, dy (128 B each), B, C (256 B each); dt, lambda 8 B; omega 256 B; fp32 dx 256, dB, dC 512 each,
    # ddt, dlambda 8, domega 256: 2576 B per (token, head), plus dA
    assert bench.bwd_bytes(w) == 2576 * th + 8 * w.heads
    assert abs(bench.FP32_ALU_TFLOPS - 148 * 128 * 2 * 2.032e9 / 1e12) < 1e-9


def test_backward_flops_grow_with_the_rank():
    bench = _bench()
    from state_space_sequence_04_b300 import synth
    import dataclasses
    w1 = synth.SISO_1P5B
    w4 = dataclasses.replace(w1, rank=4)
    assert bench.bwd_flops(w4) / bench.bwd_flops(w1) == (26 + 40) / 36
