"""The checked build (libpe_checked.so: the same entry points compiled with
PE_CHECKED, a stand-in for a sanitizer): identical outputs on valid inputs
with no error bit, PE_ERR_NAN when a logits row read by the greedy argmax
holds a NaN (vector body or scalar tail, bf16 or fp32), and no such bit from
the regular build, which leaves that precondition unchecked."""
import ctypes

import pytest
import torch

from gpu_util import Guarded, assert_same, guarded_outputs, oracle_of
from speculative_decoding_pe_gb300 import _native, build, harness
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    _native.load()
    return _native.load_checked()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _step(lib, w, early=False):
    g = Guarded()
    out = guarded_outputs(w, g)
    ws = _native.new_workspace(w.B * (w.Kp + 1), w.B)
    err = _native.new_error_word()
    args = harness.pack(w, out, ws, err)
    fn = lib.pe_step_early_exit if early else lib.pe_step
    fn.argtypes = [ctypes.POINTER(_native.StepArgs), ctypes.c_void_p]
    rc = fn(ctypes.byref(args), _stream())
    assert rc == 0, lib.pe_status_str(rc)
    torch.cuda.synchronize()
    g.check()
    res = harness.to_host(out)
    res["err"] = int(err.item())
    return res, ws


CASES = [wl.SPECS["tiny"],
         wl.SPECS["decode_b256"].with_(name="decode_small", B=24, V=30011, row_pad=5, H=128),
         wl.SPECS["prefill_b8"].with_(name="prefill_small", B=5, prompt_lo=1, prompt_hi=300,
                                      V=5003, row_pad=5, H=72)]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_checked_build_matches_oracle(checked, spec):
    w = wl.make_workload(spec, 11, device="cuda")
    ref = oracle_of(w)
    got, ws = _step(checked, w)
    assert_same(got, ref, what="checked " + spec.name)
    assert got["err"] == 0 and int(ws.count_nonzero()) == 0
    got, ws = _step(checked, w, early=True)
    keys = [k for k in harness.OUTPUT_KEYS if k != "target_argmax"] + ["err"]
    assert_same(got, ref, keys=keys, what="checked early " + spec.name)


@pytest.mark.parametrize("dtype,V,col", [(torch.bfloat16, 30011, 17),      # a vector
                                         (torch.bfloat16, 30011, 30009),   # the scalar tail
                                         (torch.float32, 1001, 1000),      # the scalar tail
                                         (torch.float32, 1001, 512)])
def test_nan_logits_raise_the_nan_bit(checked, dtype, V, col):
    pad = (-V) % (8 if dtype == torch.bfloat16 else 4)
    spec = wl.SPECS["decode_b256"].with_(name="nan", B=6, V=V, row_pad=pad, H=64, dtype=dtype)
    w = wl.make_workload(spec, 3, device="cuda")
    w.logits[2 * (w.Kp + 1) + 1, col] = float("nan")  # request 2, verified row 1
    got, _ = _step(checked, w)
    assert got["err"] & _native.ERR_NAN
    got, _ = _step(checked, w, early=True)  # row 1 is read: request 2 accepts >= 1 or
    if int(w.planted_accept[2]) >= 1:        # row 1 holds its bonus
        assert got["err"] & _native.ERR_NAN
    # verification alone and the drafter readout take the same argmax
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    bon = torch.empty(w.B, dtype=torch.int32, device="cuda")
    ws = _native.new_workspace(w.B * (w.Kp + 1), w.B)
    err = _native.new_error_word()
    rc = checked.pe_verify_greedy(w.logits.data_ptr(), _native._dtype_code(w.logits),
                                  w.logits.stride(0), w.B, w.Kp, V, w.in_tokens.data_ptr(),
                                  acc.data_ptr(), bon.data_ptr(), None, ws.data_ptr(),
                                  err.data_ptr(), _stream())
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) & _native.ERR_NAN
    # the regular build does not look for NaN
    regular = _native.load()
    got, _ = _step(regular, w)
    assert not got["err"] & _native.ERR_NAN
