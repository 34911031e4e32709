"""The single pass (one cooperative launch, one unit per CTA, chunk keys in
workspace slots) against the oracle, on both sides of the batch sizes where
the plan stops fitting, and the persistent queue on the same inputs.

With the default knob the fused step takes the single pass while every unit
fits one per co-resident CTA (decode up to about B=40 at V=201088); the
tests run each batch size with the knob on and off, so both paths are
checked on identical inputs whatever the plan decides.  pe_verify_greedy and
pe_draft_readout take the same single pass with argmax units only."""
import pytest
import torch

import oracle
from gpu_util import assert_same, oracle_of, run_fused
from speculative_decoding_pe_gb300 import _native, build
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


class knob:
    def __init__(self, single_pass):
        self.single_pass = single_pass

    def __enter__(self):
        self.before = _native.get_tuning()["single_pass"]
        _native.set_tuning(single_pass=self.single_pass)

    def __exit__(self, *exc):
        _native.set_tuning(single_pass=self.before)


# decode at V=201088 (a whole-vector vocabulary) and at V=201091 (a scalar
# tail in the last chunk); B=40-48 straddle the plan's limit
@pytest.mark.parametrize("B", [1, 2, 3, 8, 17, 40, 48])
@pytest.mark.parametrize("V", [201088, 201091])
def test_fused_step_both_paths(B, V):
    spec = wl.SPECS["decode_b1"].with_(B=B, V=V, H=256, bt_width=1025, row_pad=(-V) % 8)
    w = wl.make_workload(spec, 600 + B, device="cuda")
    ref = oracle_of(w)
    for sp in (1, -1):
        with knob(sp):
            assert_same(run_fused(w), ref, what="B=%d V=%d single_pass=%d" % (B, V, sp))


@pytest.mark.parametrize("B", [1, 4, 8])
def test_verify_both_paths(B):
    w = wl.make_workload(wl.SPECS["decode_b1"].with_(B=B, H=64, bt_width=1025), 700 + B,
                         device="cuda")
    rows = B * (w.Kp + 1)
    ref = oracle_of(w)
    for sp in (1, -1):
        with knob(sp):
            acc = torch.empty(B, dtype=torch.int32, device="cuda")
            bon = torch.empty_like(acc)
            amax = torch.empty(rows, dtype=torch.int32, device="cuda")
            ws = _native.new_workspace(rows, B)
            err = _native.new_error_word()
            _native.verify_greedy(w.logits, w.Kp, w.in_tokens, acc, bon, ws, err,
                                  target_argmax=amax)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert torch.equal(acc.cpu(), ref["accepted_len"].to(torch.int32)), sp
            assert torch.equal(bon.cpu(), ref["bonus_token"].to(torch.int32)), sp
            assert torch.equal(amax.cpu(), ref["target_argmax"].to(torch.int32)), sp
            assert int(ws.count_nonzero()) == 0


# 7 rows (one request), 112, and 1100 rows (more units than the slots hold)
@pytest.mark.parametrize("n", [7, 112, 1100])
def test_readout_both_paths(n):
    g = torch.Generator().manual_seed(800 + n)
    V = 151936
    logits = (torch.randn(n, V, generator=g) * 2).to(torch.bfloat16)
    ref = oracle.argmax_rows(logits)
    dev = logits.cuda()
    for sp in (1, -1):
        with knob(sp):
            out = torch.empty(n, dtype=torch.int32, device="cuda")
            ws = _native.new_workspace(n, n)
            err = _native.new_error_word()
            _native.draft_readout(dev, out, ws, err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert torch.equal(out.cpu(), ref.to(torch.int32)), sp
            assert int(ws.count_nonzero()) == 0
