"""Early-exit verification (pe_step_early_exit) against the CPU oracle.

Every output must equal the full step's bit for bit, except target_argmax:
rows 0..a_b of each request carry their argmax, later rows -1 (they may
never have been read).  Every test runs twice: with the early-exit kernel
forced, and with the default, under which small batches (logits of at most
pe_tuning.early_full_read_mb MiB) are served by the full-read kernel with
the same outputs."""
import pytest
import torch

import pins
from gpu_util import Guarded, assert_same, guarded_outputs, oracle_of
from speculative_decoding_pe_gb300 import _native, build, harness
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


def _restore(t):
    _native.set_tuning(**{k: (v if v or k != "early_full_read_mb" else -1) for k, v in t.items()})


@pytest.fixture(autouse=True, params=["early_kernel", "default"])
def early_path(request):
    before = _native.get_tuning()
    _native.set_tuning(early_full_read_mb=-1 if request.param == "early_kernel" else 128)
    yield request.param
    _restore(before)


def run_early(w, workspace=None):
    g = Guarded()
    out = guarded_outputs(w, g)
    ws = workspace if workspace is not None else _native.new_workspace(w.B * (w.Kp + 1), w.B)
    err = _native.new_error_word()
    harness.run(w, out, ws, err, early_exit=True)
    torch.cuda.synchronize()
    g.check()
    assert int(ws.count_nonzero()) == 0, "workspace not left zeroed"
    res = harness.to_host(out)
    res["err"] = int(err.item())
    return res, ws


def check_early(w, got, ref):
    keys = [k for k in harness.OUTPUT_KEYS if k != "target_argmax"] + ["err"]
    assert_same(got, ref, keys=keys, what=w.spec.name + " early exit")
    nr = w.Kp + 1
    ta = got["target_argmax"].view(w.B, nr)
    ra = ref["target_argmax"].view(w.B, nr)
    for b in range(w.B):
        a = int(ref["accepted_len"][b])
        assert torch.equal(ta[b, :a + 1], ra[b, :a + 1]), b
        assert (ta[b, a + 1:] == -1).all(), b


FULL = [("tiny", 0), ("tiny", 1), ("decode_b1", 0), ("decode_b64", 0), ("prefill_b8", 0),
        ("decode_b256", 0), ("decode_b256", 1)]


@pytest.mark.parametrize("name,trial", FULL, ids=lambda v: str(v))
def test_early_exit_full_size(name, trial):
    cfg = list(wl.SPECS).index(name) + 1
    w = wl.make_workload(name, 1000 * cfg + trial, device="cuda")
    got, ws = run_early(w)
    check_early(w, got, oracle_of(w))


@pytest.mark.parametrize("spec", pins._small_specs() + [
    wl.SPECS["decode_b256"].with_(name="all_accept", B=40, forced=tuple((b, 7) for b in range(40))),
    wl.SPECS["decode_b256"].with_(name="none_accept", B=40, forced=tuple((b, 0) for b in range(40))),
    wl.SPECS["decode_b256"].with_(name="ragged", B=30, V=151937, row_pad=7, H=256),
    wl.SPECS["decode_b256"].with_(name="kp31", B=9, Kp=31, K=4, V=4099, row_pad=5, H=64,
                                  accept_p=0.05),
], ids=lambda s: s.name)
def test_early_exit_variants(spec):
    for seed in (0, 1):
        w = wl.make_workload(spec, seed, device="cuda")
        got, _ = run_early(w)
        check_early(w, got, oracle_of(w))


@pytest.mark.parametrize("queue_order", [1, 2], ids=["tiles_first", "tiles_last"])
def test_early_exit_queue_orders(queue_order):
    """Either order of copy tiles and argmax chunks gives the same outputs:
    the bonus row is written by the verdict or by the request's last
    verified-row tile, whichever comes second."""
    before = _native.get_tuning()
    try:
        _native.set_tuning(queue_order=queue_order, rows_per_unit=3)
        for spec, seed in ((wl.SPECS["decode_b256"].with_(B=48, V=30011, row_pad=5), 11),
                           (wl.SPECS["decode_b64"].with_(B=16, V=20011, row_pad=5), 12)):
            w = wl.make_workload(spec, seed, device="cuda")
            got, ws = run_early(w)
            check_early(w, got, oracle_of(w))
            assert int(ws.count_nonzero()) == 0
    finally:
        _native.set_tuning(**before)


def test_workspace_shared_with_full_step():
    """Early-exit and full steps alternate on one workspace; each leaves it
    clean for the other."""
    ws = _native.new_workspace(256 * 8, 256)
    for i in range(6):
        w = wl.make_workload(wl.SPECS["decode_b256"].with_(B=64 + 32 * i, V=30011, row_pad=5),
                             300 + i, device="cuda")
        ref = oracle_of(w)
        if i % 2:
            got, _ = run_early(w, ws)
            check_early(w, got, ref)
        else:
            out, _, err = harness.allocate(w)
            harness.run(w, out, ws, err)
            torch.cuda.synchronize()
            got = harness.to_host(out)
            got["err"] = int(err.item())
            assert_same(got, ref)
        assert int(ws.count_nonzero()) == 0, i


def test_kp_above_31_rejected():
    w = wl.make_workload(wl.SPECS["tiny"].with_(Kp=32, K=2, B=2, V=101, row_pad=3), 0,
                         device="cuda")
    out, ws, err = harness.allocate(w)
    with pytest.raises(_native.PEError):
        harness.run(w, out, ws, err, early_exit=True)


def test_early_mismatch_edges():
    """Rows where a chunk can tell the row's argmax is not the draft before
    the row completes, and rows where it must not: a draft outside the
    vocabulary (never the argmax), the row maximum repeated at a column
    below the draft (the argmax is that column: a mismatch) and above it
    (the draft keeps the argmax).  Each row spans two chunks, so a chunk can
    end before its row completes."""
    spec = wl.SPECS["decode_b256"].with_(B=48, V=60011, row_pad=5, H=64)
    w = wl.make_workload(spec, 77)
    nr = w.Kp + 1
    g = torch.Generator().manual_seed(5)
    acc = w.planted_accept.tolist()
    for b in range(w.B):
        a = int(acc[b])
        kind = b % 4
        if a == 0 or kind == 0:
            continue
        j = int(torch.randint(0, a, (1,), generator=g))  # a matching row
        row = b * nr + j
        d = int(w.in_tokens[b * nr + j + 1])
        if kind == 1:    # the draft outside the vocabulary: a mismatch at row j
            w.in_tokens[b * nr + j + 1] = w.V + 5 if b % 8 == 1 else -3
        elif kind == 2:  # the maximum also at a lower column: a mismatch
            if d > 0:
                w.logits[row, d - 1 - int(torch.randint(0, d, (1,), generator=g))] = w.logits[row, d]
        else:            # the maximum also at a higher column: still a match
            if d < w.V - 1:
                c = d + 1 + int(torch.randint(0, w.V - 1 - d, (1,), generator=g))
                w.logits[row, c] = w.logits[row, d]
    wg = w.to("cuda")
    ref = oracle_of(wg)
    got, _ = run_early(wg)
    check_early(wg, got, ref)
