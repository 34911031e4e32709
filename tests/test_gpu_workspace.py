"""A workspace that was not zero when a call started is detected, never
followed out of bounds, and a re-zeroed workspace serves the next call.

Every entry point that takes a workspace assumes it is zero and leaves it
zero.  Here one word of a zeroed workspace at a time is overwritten on the
host with a value no legal call leaves there (0xA5 bytes; for a row key, a
value above every real key whose column lies outside the vocabulary), the
call runs, and PE_ERR_WORKSPACE must be raised.  The outputs of that call
are not checked (the bit says they are incomplete); the guard bands around
them are, so a stray write would still fail.  The workspace is then zeroed
again and the next call must equal the oracle bit for bit with no error bit.
Nothing here waits on another CTA, so none of these calls can hang.

The word offsets restate the layouts documented beside the kernels
(pe_workspace.cuh; the sampled layout in pe_sampled.cu)."""
import pytest
import torch

import oracle
from gpu_util import Guarded, assert_same, guarded_outputs, oracle_of
from speculative_decoding_pe_gb300 import _native, build, harness
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

U32 = 0xA5A5A5A5
U64 = 0xA5A5A5A5A5A5A5A5
KEY = 0xFFFFFFFFA5A5A5A5  # beats every real key; column 0x5A5A5A5A >= V


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


def _greedy_offsets(rows, B):
    """Byte offsets of the greedy workspace's fields (pe_workspace.cuh)."""
    count = 8
    state = (count + 4 * B + 7) & ~7
    xfer = state + 8 * B
    key = xfer + 8 * B
    rcount = key + 8 * rows
    amax = rcount + 4 * rows
    slot = (amax + 4 * rows + 7) & ~7
    return {"sched": 0, "ctas_done": 4, "count": count, "state": state, "xfer": xfer,
            "key": key, "rcount": rcount, "slot": slot}


def _poke(ws, offset, value, nbytes):
    ws[offset:offset + nbytes] = torch.tensor(
        list(int(value).to_bytes(nbytes, "little")), dtype=torch.uint8, device=ws.device)


def _run(w, ws, early):
    g = Guarded()
    out = guarded_outputs(w, g)
    err = _native.new_error_word()
    harness.run(w, out, ws, err, early_exit=early)
    torch.cuda.synchronize()
    g.check()
    res = harness.to_host(out)
    res["err"] = int(err.item())
    return res


class tuned:
    def __init__(self, **kw):
        self.kw = kw

    def __enter__(self):
        self.before = _native.get_tuning()
        _native.set_tuning(**self.kw)

    def __exit__(self, *exc):
        b = dict(self.before)
        if b["early_full_read_mb"] == 0:
            b["early_full_read_mb"] = -1
        _native.set_tuning(**b)


# B=8, K'=7, V=151936: 64 rows of about ten chunks each, so per-row and
# per-request counts both matter
SPEC = wl.SPECS["decode_b256"].with_(B=8, H=256, bt_width=4097)

# (field, byte offset within the field, bytes, value); request 1, row 8 =
# request 1's row 0 (read by every path, early exit included)
FULL_CASES = [("sched", 0, 4, U32), ("count", 4, 4, U32), ("xfer", 8, 8, U64),
              ("key", 8 * 8, 8, KEY)]
EARLY_CASES = [("sched", 0, 4, U32), ("ctas_done", 0, 4, U32), ("state", 8, 8, U64),
               ("rcount", 4 * 8, 4, U32), ("key", 8 * 8, 8, KEY), ("xfer", 8, 8, U64),
               ("count", 4, 4, U32)]  # early exit: request 1's early-mismatch word


@pytest.mark.parametrize("variant", [1, 2], ids=["regs", "bulk"])
@pytest.mark.parametrize("field,off,nbytes,value", FULL_CASES, ids=[c[0] for c in FULL_CASES])
def test_fused_step_detects_dirty_workspace(field, off, nbytes, value, variant):
    w = wl.make_workload(SPEC, 41, device="cuda")
    ref = oracle_of(w)
    rows = w.B * (w.Kp + 1)
    ws = _native.new_workspace(rows, w.B)
    _poke(ws, _greedy_offsets(rows, w.B)[field] + off, value, nbytes)
    with tuned(variant=variant, single_pass=-1):  # the persistent queue, which uses them
        got = _run(w, ws, early=False)
        assert got["err"] & _native.ERR_WORKSPACE, field
        ws.zero_()
        again = _run(w, ws, early=False)
    assert_same(again, ref, what="after re-zeroing (%s)" % field)
    assert int(ws.count_nonzero()) == 0


@pytest.mark.parametrize("slot", [0, 7, 63], ids=["first", "second", "later_request"])
def test_single_pass_detects_a_dirty_slot(slot):
    """A few requests run as a single pass: each argmax unit stores its chunk
    key into its own slot and the request's last chunk collects them.  A slot
    left holding a value no chunk of this step can store is either
    overwritten by its chunk before the collector reads it (the outputs are
    then exact) or read first and reported; it is never taken silently."""
    w = wl.make_workload(SPEC, 44, device="cuda")
    ref = oracle_of(w)
    rows = w.B * (w.Kp + 1)
    ws = _native.new_workspace(rows, w.B)
    _poke(ws, _greedy_offsets(rows, w.B)["slot"] + 8 * slot, KEY, 8)
    got = _run(w, ws, early=False)
    if not got["err"] & _native.ERR_WORKSPACE:
        assert_same(got, ref, what="dirty slot %d overwritten in time" % slot)
    ws.zero_()
    again = _run(w, ws, early=False)
    assert_same(again, ref, what="after re-zeroing (slot %d)" % slot)
    assert int(ws.count_nonzero()) == 0


@pytest.mark.parametrize("field,off,nbytes,value", EARLY_CASES, ids=[c[0] for c in EARLY_CASES])
def test_early_exit_detects_dirty_workspace(field, off, nbytes, value):
    w = wl.make_workload(SPEC, 42, device="cuda")
    ref = oracle_of(w)
    ref["target_argmax"] = ref["target_argmax"].clone()
    for b in range(w.B):  # early exit reports -1 for rows after a_b
        a = int(ref["accepted_len"][b])
        ref["target_argmax"][b * (w.Kp + 1) + a + 1:(b + 1) * (w.Kp + 1)] = -1
    rows = w.B * (w.Kp + 1)
    ws = _native.new_workspace(rows, w.B)
    _poke(ws, _greedy_offsets(rows, w.B)[field] + off, value, nbytes)
    with tuned(early_full_read_mb=-1):  # the early-exit kernel, not the full read
        got = _run(w, ws, early=True)
        assert got["err"] & _native.ERR_WORKSPACE, field
        ws.zero_()
        again = _run(w, ws, early=True)
    assert_same(again, ref, what="after re-zeroing (%s)" % field)
    assert int(ws.count_nonzero()) == 0


def test_verify_and_readout_detect_dirty_workspace():
    with tuned(single_pass=-1):  # the persistent queue, which uses these words
        _verify_and_readout_detect_dirty_workspace()


def _verify_and_readout_detect_dirty_workspace():
    w = wl.make_workload(SPEC, 43, device="cuda")
    rows = w.B * (w.Kp + 1)
    ref = oracle.argmax_rows(w.logits.cpu())
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    bon = torch.empty_like(acc)
    amax = torch.empty(rows, dtype=torch.int32, device="cuda")
    for field, off, nbytes, value in FULL_CASES[:2] + FULL_CASES[3:]:
        ws = _native.new_workspace(rows, w.B)
        _poke(ws, _greedy_offsets(rows, w.B)[field] + off, value, nbytes)
        err = _native.new_error_word()
        _native.verify_greedy(w.logits, w.Kp, w.in_tokens, acc, bon, ws, err,
                              target_argmax=amax)
        torch.cuda.synchronize()
        assert int(err.item()) & _native.ERR_WORKSPACE, field
        ws.zero_()
        err.zero_()
        _native.verify_greedy(w.logits, w.Kp, w.in_tokens, acc, bon, ws, err,
                              target_argmax=amax)
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and torch.equal(amax.cpu(), ref), field
        assert int(ws.count_nonzero()) == 0
    # readout: n sampled rows, each its own request of one row
    n = rows
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    ws = _native.new_workspace(n, n)
    _poke(ws, _greedy_offsets(n, n)["key"] + 8 * 5, KEY, 8)
    err = _native.new_error_word()
    _native.draft_readout(w.logits, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & _native.ERR_WORKSPACE
    ws.zero_()
    err.zero_()
    _native.draft_readout(w.logits, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and torch.equal(out.cpu(), ref)


# ------------------------------------------------------- rejection sampling

def _sampled_offsets(B, Kp):
    """Byte offsets of the sampled workspace's fields (pe_sampled.cu)."""
    rows = B * (Kp + 1) + B * Kp
    o = 32 + 4 * 64 * 2
    offs = {}

    def take(name, n):
        nonlocal o
        o = (o + 15) // 16 * 16
        offs[name] = o
        o += n
    take("partial", 8 * rows * 32)
    take("lse", 4 * rows)
    take("prob", 4 * rows)
    take("rcount", 4 * rows)
    take("qcount", 4 * B)
    take("dcount", 4 * B)
    take("acc", 4 * B)
    take("gkey", 8 * B)
    take("rkey", 8 * B)
    take("rlist", 4 * B)
    offs.update({"residual_done": 12, "listed": 16, "stats_counter0": 32,
                 "stats_counter1": 32 + 256})
    return offs


def _sampled(s, ws, T, seed):
    acc = torch.empty(s.B, dtype=torch.int32, device="cuda")
    bon = torch.empty_like(acc)
    err = _native.new_error_word()
    _native.verify_sampled(s.target_logits, s.draft_logits, s.Kp, s.tokens, s.u_accept, T,
                           seed, acc, bon, ws, err)
    torch.cuda.synchronize()
    return acc.cpu(), bon.cpu(), int(err.item())


def test_sampled_verification_detects_dirty_workspace():
    B, Kp, V, T, seed = 8, 3, 20000, 1.0, 77
    host = wl.make_sampled_inputs(B, Kp, V, seed=5)
    s = host.to("cuda")
    ref_acc, ref_bon = oracle.verify_sampled(host.target_logits, host.draft_logits, B, Kp,
                                             host.tokens, host.u_accept, T, seed)
    nbytes = _native.workspace_bytes_sampled(B, Kp)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    acc, bon, err = _sampled(s, ws, T, seed)
    assert err == 0 and torch.equal(acc, ref_acc) and torch.equal(bon, ref_bon)
    rejecting = [b for b in range(B) if int(ref_acc[b]) < Kp]
    assert rejecting, "the inputs must hold a rejection"
    rb = rejecting[0]
    offs = _sampled_offsets(B, Kp)
    cases = [("stats_counter0", 0, 4, U32), ("stats_counter1", 0, 4, U32),
             ("residual_done", 0, 4, U32), ("listed", 0, 4, U32),
             ("rcount", 0, 4, U32), ("qcount", 4 * 1, 4, U32),
             ("dcount", 4 * rb, 4, U32), ("gkey", 8 * 1, 8, KEY), ("rkey", 8 * rb, 8, KEY)]
    for field, off, nb, value in cases:
        ws.zero_()
        _poke(ws, offs[field] + off, value, nb)
        _, _, err = _sampled(s, ws, T, seed)
        assert err & _native.ERR_WORKSPACE, field
        ws.zero_()
        acc, bon, err = _sampled(s, ws, T, seed)
        assert err == 0 and torch.equal(acc, ref_acc) and torch.equal(bon, ref_bon), field
        assert int(ws.count_nonzero()) == 0, field
