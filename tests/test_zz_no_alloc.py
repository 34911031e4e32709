"""pe_step_noalloc: the fused step for callers that cannot allocate device
memory (a runtime whose pool owns the whole device, a plug-in that only sees
its tensors, a loop that must not hit cudaMalloc's device synchronisation).
Its scratch is a fixed array inside the library instead of a caller
workspace.  Called here through the C ABI and compared bit for bit with the
CPU oracle (and with pe_step) on the same inputs, several calls in a row on
one stream, so that each call sees whatever the one before it left in the
shared array: a large batch after a small one, and the same batch twice.

This file is named to be collected last; it passes alone in a fresh process
as well as after the other tests."""
import ctypes

import pytest
import torch

from gpu_util import assert_same, oracle_of
from speculative_decoding_pe_gb300 import _native, build, harness
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _with_pe_step(w):
    out, ws, err = harness.allocate(w)
    harness.run(w, out, ws, err)
    return out, err


def _noalloc(lib, w):
    out, ws, err = harness.allocate(w)
    args = harness.pack(w, out, ws, err)
    args.workspace = None            # ignored by this entry point
    rc = lib.pe_step_noalloc(ctypes.byref(args), _stream())
    assert rc == 0, lib.pe_status_str(rc)
    return out, err


def _host(out, err):
    h = harness.to_host(out)
    h["err"] = int(err.item())
    return h


def test_noalloc_matches_the_oracle_calls_in_a_row(lib):
    small = wl.make_workload(wl.SPECS["prefill_b8"].with_(B=1, prompt_lo=3, prompt_hi=40,
                                                          V=2003, row_pad=5, H=64),
                             30, device="cuda")
    big = wl.make_workload("decode_b256", 31, device="cuda")
    mid = wl.make_workload(wl.SPECS["prefill_b8"].with_(B=5, prompt_lo=1, prompt_hi=600,
                                                        V=5003, row_pad=5, H=72),
                           32, device="cuda")
    cases = [small, big, mid, big]   # a B=1, K'=0 call first, then B=256 ...
    got = [_noalloc(lib, w) for w in cases]   # one stream, no synchronisation between
    torch.cuda.synchronize()
    refs = {id(w): oracle_of(w) for w in (small, big, mid)}
    for w, g in zip(cases, got):
        assert_same(_host(*g), refs[id(w)], what="noalloc " + w.spec.name)
    # the same outputs as pe_step with a caller workspace
    for w in (small, big):
        assert_same(_host(*_with_pe_step(w)), refs[id(w)], what="pe_step " + w.spec.name)


def test_noalloc_allocates_nothing(lib):
    w = wl.make_workload("decode_b256", 33, device="cuda")
    out, ws, err = harness.allocate(w)
    args = harness.pack(w, out, ws, err)
    args.workspace = None
    for _ in range(2):  # the first call may load the library's GPU code
        assert lib.pe_step_noalloc(ctypes.byref(args), _stream()) == 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    allocated_before = torch.cuda.memory_allocated()
    assert lib.pe_step_noalloc(ctypes.byref(args), _stream()) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.cuda.memory_allocated() == allocated_before
    assert_same(_host(out, err), oracle_of(w), what="noalloc decode_b256")


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    too_big = wl.SPECS["decode_b256"].with_(B=1024, V=64, H=8, bt_width=4097)
    w = wl.make_workload(too_big, 1, device="cuda")
    assert lib.pe_workspace_bytes(w.B * (w.Kp + 1), w.B) > 65536
    out, ws, err = harness.allocate(w)
    args = harness.pack(w, out, ws, err)
    args.workspace = None
    assert lib.pe_step_noalloc(ctypes.byref(args), _stream()) == -1   # PE_EINVAL
    assert lib.pe_step_noalloc(None, _stream()) == -1
