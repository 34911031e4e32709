"""The fused step inside a captured CUDA graph: several steps with their own
inputs and outputs, one shared workspace, replayed more than once.  Every
replay must give the oracle's outputs bit for bit and leave the workspace
zeroed (the entry points allocate nothing, never synchronise, and read
device attributes once, on their first call, which comes before capture)."""
import pytest
import torch

from gpu_util import assert_same, oracle_of
from speculative_decoding_pe_gb300 import _native, build, harness
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


@pytest.mark.parametrize("early_exit", [False, True], ids=["full", "early_exit"])
@pytest.mark.parametrize("name", ["decode_b64", "prefill_b8", "tiny"])
def test_steps_captured_in_one_graph(name, early_exit):
    spec = wl.SPECS[name]
    if name == "decode_b64":
        spec = spec.with_(B=32, V=50021, row_pad=3)
    if name == "prefill_b8":
        spec = spec.with_(B=4, prompt_lo=10, prompt_hi=500, V=20011, row_pad=5, H=64)
    steps = [wl.make_workload(spec, 40 + i, device="cuda") for i in range(3)]
    ws = _native.new_workspace(max(w.logits_rows for w in steps), max(w.B for w in steps))
    run = _native.step_early_exit_packed if early_exit else _native.step_packed
    bufs = [harness.allocate(w) for w in steps]
    packed = [harness.pack(w, out, ws, err) for w, (out, _, err) in zip(steps, bufs)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(packed[0], s)            # first call: device attributes, before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for a in packed:
            run(a, torch.cuda.current_stream())
    for _ in range(2):
        for out, _, err in bufs:
            out.X.fill_(7)
            err.zero_()
        g.replay()
        torch.cuda.synchronize()
        for w, (out, _, err) in zip(steps, bufs):
            got = harness.to_host(out)
            got["err"] = int(err.item())
            ref = oracle_of(w)
            keys = [k for k in harness.OUTPUT_KEYS if not (early_exit and k == "target_argmax")]
            assert_same(got, ref, keys=keys + ["err"], what=name)
        assert int(ws.count_nonzero()) == 0


def test_sampled_verification_captured_in_one_graph():
    """pe_verify_sampled (a stats launch, then the residual launch as its
    programmatic dependent) captured twice with distinct inputs and one
    workspace; every replay equals the same calls made eagerly."""
    cases = [wl.make_sampled_inputs(24, 5, 20011, seed=60 + i).to("cuda") for i in range(2)]
    ws = torch.zeros(_native.workspace_bytes_sampled(24, 5), dtype=torch.uint8, device="cuda")
    outs = [(torch.empty(24, dtype=torch.int32, device="cuda"),
             torch.empty(24, dtype=torch.int32, device="cuda"), _native.new_error_word())
            for _ in cases]

    def call(i, stream):
        s, (acc, bon, err) = cases[i], outs[i]
        _native.verify_sampled(s.target_logits, s.draft_logits, s.Kp, s.tokens, s.u_accept,
                               0.9, 77 + i, acc, bon, ws, err, stream)

    for i in range(2):  # eager results (and the first call on the device)
        call(i, None)
    torch.cuda.synchronize()
    ref = [(a.clone(), b.clone()) for a, b, _ in outs]
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for i in range(2):
            call(i, torch.cuda.current_stream())
    for _ in range(2):
        for acc, bon, err in outs:
            acc.fill_(-5)
            bon.fill_(-5)
            err.zero_()
        g.replay()
        torch.cuda.synchronize()
        for (acc, bon, err), (ra, rb) in zip(outs, ref):
            assert int(err.item()) == 0
            assert torch.equal(acc, ra) and torch.equal(bon, rb)
        assert int(ws.count_nonzero()) == 0
