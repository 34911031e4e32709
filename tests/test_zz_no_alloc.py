"""pe_step_noalloc: the fused step for callers that cannot allocate device
memory (a runtime whose pool owns the whole device, a plug-in that only sees
its tensors, a loop that must not hit cudaMalloc's device synchronisation).
Its scratch is a fixed array inside the library instead of a caller
workspace.  Called here through the C ABI and compared bit for bit with
pe_step on the same inputs, two calls in a row, so that a second call sees
whatever the first one left in the shared array.

This file is named to be collected last; it passes alone in a fresh process
as well as after the other tests."""
import ctypes

import pytest
import torch

from gpu_util import assert_same
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


def _reference(w):
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


def test_noalloc_matches_pe_step_two_calls_in_a_row(lib):
    cases = [wl.make_workload("decode_b256", 31, device="cuda"),
             wl.make_workload(wl.SPECS["prefill_b8"].with_(B=5, prompt_lo=1, prompt_hi=600,
                                                           V=5003, row_pad=5, H=72),
                              32, device="cuda")]
    refs = [_reference(w) for w in cases]
    # two calls in a row on one stream, no synchronisation in between
    got = [_noalloc(lib, w) for w in cases]
    torch.cuda.synchronize()
    for w, r, g in zip(cases, refs, got):
        assert_same(_host(*g), _host(*r), what="noalloc " + w.spec.name)
    # and the same workload twice: the second call starts from what the
    # first one left in the shared scratch
    again = [_noalloc(lib, cases[0]) for _ in range(2)]
    torch.cuda.synchronize()
    for g in again:
        assert_same(_host(*g), _host(*refs[0]), what="noalloc repeat")


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    too_big = wl.SPECS["decode_b256"].with_(B=1024, V=64, H=8, bt_width=4097)
    w = wl.make_workload(too_big, 1, device="cuda")
    assert lib.pe_workspace_bytes(w.B * (w.Kp + 1), w.B) > 65536
    out, ws, err = harness.allocate(w)
    args = harness.pack(w, out, ws, err)
    args.workspace = None
    assert lib.pe_step_noalloc(ctypes.byref(args), _stream()) == -1   # PE_EINVAL
    assert lib.pe_step_noalloc(None, _stream()) == -1
