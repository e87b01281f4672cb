"""Host-side tests of the C ABI: the library loads without a GPU, exports every
symbol include/m3.h declares, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import pytest

from state_space_sequence_04_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"M3_API\s+[\w\s\*]+?\b(m3_\w+)\s*\(", txt)
    return names


@pytest.fixture(scope="module")
def lib():
    from state_space_sequence_04_b300 import build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    return binding.load()


def test_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert len(names) >= 6
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(binding.SIGNATURES), "binding lacks a signature for a declared symbol"


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        s = binding.m3_status_string(code)
        assert s.startswith("M3_")
    assert binding.m3_status_string(-99) == "unknown m3 status"
    assert binding.m3_version() >= 100


def _scan(lib, ptrs=None, **kw):
    d = dict(R=1, chunk=64, Bt=1, T=128, H=2, P=64, N=128, io=0, ws=None, ws_bytes=0)
    d.update(kw)
    p = dict(x=16, B=32, C=48, dt=64, A=80, lam=96, om=112, y=128, fin=None)
    if ptrs:
        p.update(ptrs)
    return lib.m3_scan_fwd(p["x"], p["B"], p["C"], p["dt"], p["A"], p["lam"], p["om"], d["R"], d["chunk"],
                           p["y"], p["fin"], d["Bt"], d["T"], d["H"], d["P"], d["N"], d["io"], d["ws"],
                           d["ws_bytes"], None)


def test_scan_rejects_bad_arguments(lib):
    INV, UNS, WS = binding.M3_ERR_INVALID_ARG, binding.M3_ERR_UNSUPPORTED, binding.M3_ERR_WORKSPACE
    assert _scan(lib, ptrs={"x": None}) == INV                  # null input
    assert _scan(lib, ptrs={"B": 33}) == INV                    # misaligned
    assert _scan(lib, ptrs={"fin": 8}) == INV                   # misaligned optional output
    assert _scan(lib, N=127) == INV                             # odd state size
    assert _scan(lib, io=7) == INV                              # unknown dtype
    assert _scan(lib, Bt=-1) == INV
    assert _scan(lib, R=3) == UNS                               # rank not implemented
    assert _scan(lib, chunk=24) == UNS                          # chunk not a multiple of 16
    assert _scan(lib, chunk=512) == UNS
    assert _scan(lib, P=12) == UNS
    assert _scan(lib, N=1024) == UNS
    # workspace: required size is positive for this shape, so none / too small / misaligned fail
    need = binding.m3_scan_fwd_workspace_size(1, 128, 2, 64, 128, 1, 64, 0)
    assert need > 0
    assert _scan(lib) == WS
    assert _scan(lib, ws=1 << 20, ws_bytes=need - 1) == WS
    assert _scan(lib, ws=(1 << 20) + 16, ws_bytes=need) == WS
    assert binding.m3_scan_fwd_workspace_size(1, 128, 2, 64, 127, 1, 64, 0) == 0


def test_scan_empty_batch_is_noop(lib):
    # batch 0: valid, nothing launched, no workspace needed
    assert binding.m3_scan_fwd_workspace_size(0, 128, 2, 64, 128, 1, 64, 0) == 0
    assert _scan(lib, Bt=0, ptrs={"x": None, "B": None, "C": None, "y": None}) == binding.M3_OK


def test_decode_rejects_bad_arguments(lib):
    INV, UNS = binding.M3_ERR_INVALID_ARG, binding.M3_ERR_UNSUPPORTED

    def dec(R=1, b=2, H=2, P=64, N=128, io=0, **ptrs):
        p = dict(state=16, x=32, B=48, cache=64, C=80, dt=96, A=112, lam=128, om=144, y=160)
        p.update(ptrs)
        return lib.m3_decode_step(p["state"], p["x"], p["B"], p["cache"], p["C"], p["dt"], p["A"], p["lam"],
                                  p["om"], p["y"], b, H, P, N, R, io, None)

    assert dec(state=None) == INV
    assert dec(cache=20) == INV
    assert dec(N=63) == INV
    assert dec(io=5) == INV
    assert dec(R=3) == UNS
    assert dec(R=16) == UNS
    assert dec(P=6) == UNS
    assert dec(b=0, state=None, x=None) == binding.M3_OK      # empty batch: nothing to do


def test_state_passing_rejects_bad_arguments(lib):
    INV, UNS = binding.M3_ERR_INVALID_ARG, binding.M3_ERR_UNSUPPORTED

    def sp(b=1, H=2, nc=4, N=16, P=8, S=16, ld=32, ang=48, init=None, fin=None):
        return lib.m3_state_passing(S, ld, ang, init, fin, b, H, nc, N, P, None)

    assert sp(S=None) == INV
    assert sp(ld=36) == INV
    assert sp(init=8) == INV
    assert sp(N=15) == INV
    assert sp(P=6) == INV
    assert sp(nc=-1) == INV
    assert sp(N=512) == UNS
    assert sp(b=0, S=None, ld=None, ang=None) == binding.M3_OK
