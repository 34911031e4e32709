"""The CUDA path against the CPU oracle, bit for bit (tolerance 0: every
output is an index, a copy or an argmax).

Full-size cases run the five workload shapes in the launch configuration the
benchmark uses; the oracle computes every output of them.  Smaller cases
cover the corner cases: all / none accepted, K = 1, K' = 1, prefill with
one-row prompts, ragged vocabularies (a scalar tail after the last 16-byte
vector), padded logits rows, ties across chunk boundaries, -0.0 vs +0.0,
a bonus equal to the MASK id, data errors, workspace reuse.
"""
import pytest
import torch

import oracle
import pins
from gpu_util import Guarded, assert_same, guarded_outputs, oracle_of, run_fused
from speculative_decoding_pe_gb300 import _native, build, harness
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


def _gen(spec, seed):
    return wl.make_workload(spec, seed, device="cuda")


class tuned:
    """Run a block under other launch-shape knobs, then restore them."""
    def __init__(self, **kw):
        self.kw = kw

    def __enter__(self):
        self.before = _native.get_tuning()
        _native.set_tuning(**self.kw)

    def __exit__(self, *exc):
        _native.set_tuning(**self.before)


# copy tiles through registers / bulk copies; verified-row tiles first
# (queue_order 1: the verdict usually writes the bonus row) or every tile
# after the argmax chunks (2, the default: the tiles usually write it)
VARIANTS = [dict(variant=1, queue_order=1), dict(variant=2, queue_order=1),
            dict(variant=1, queue_order=2), dict(variant=2, queue_order=2)]
VARIANT_IDS = ["regs_vfirst", "bulk_vfirst", "regs", "bulk"]


# ------------------------------------------------------------ full sizes

FULL = [("tiny", s) for s in range(4)] + [("decode_b1", 0), ("decode_b1", 1),
                                          ("decode_b64", 0), ("prefill_b8", 0),
                                          ("decode_b256", 0)]


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("name,trial", FULL, ids=lambda v: str(v))
def test_fused_step_full_size(name, trial, variant):
    cfg = list(wl.SPECS).index(name) + 1
    w = _gen(name, 1000 * cfg + trial)
    with tuned(**variant):
        got = run_fused(w)
    ref = oracle_of(w)
    assert_same(got, ref, what=name)
    if not w.spec.prefill:  # the planted lengths are what any verifier must find
        assert torch.equal(got["accepted_len"], w.planted_accept)


# ------------------------------------------------------------ small shapes

def _variants():
    out = []
    for spec in pins._small_specs():
        out.append(spec)
        if spec.dtype == torch.float32:
            pad = (8 - spec.V % 8) % 8 + (8 if spec.row_pad else 0)
            out.append(spec.with_(name=spec.name + "_bf16", dtype=torch.bfloat16,
                                  row_pad=pad))
    base = wl.SPECS["decode_b256"]
    out += [
        base.with_(name="ragged_bf16", B=6, V=151937, row_pad=7, H=256),
        base.with_(name="ragged_small", B=3, V=13, row_pad=3, H=8, bt_width=4097),
        wl.SPECS["tiny"].with_(name="ragged_f32", V=1001, row_pad=3, B=5),
        wl.SPECS["tiny"].with_(name="v_below_vector", V=3, row_pad=1, B=4),
        base.with_(name="many_requests", B=700, V=4099, row_pad=5, H=64, Kp=3, K=5),
        wl.SPECS["prefill_b8"].with_(name="prefill_small", B=13, prompt_lo=1,
                                     prompt_hi=300, V=5003, row_pad=5, H=72),
        wl.SPECS["prefill_b8"].with_(name="prefill_one_row", B=9, prompt_lo=1,
                                     prompt_hi=1, V=777, row_pad=7, H=8, K=1),
    ]
    return out


@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("spec", _variants(), ids=lambda s: s.name)
def test_fused_step_variants(spec, variant):
    for seed in (0, 1):
        w = _gen(spec, seed)
        with tuned(**variant):
            got = run_fused(w)
        assert_same(got, oracle_of(w), what=spec.name)


@pytest.mark.parametrize("tuning", [dict(), dict(ctas_per_sm=1), dict(chunk_batches=1),
                                    dict(ctas_per_sm=2, chunk_batches=2, rows_per_unit=16),
                                    dict(rows_per_unit=1),
                                    dict(variant=2, ctas_per_sm=1),
                                    dict(variant=2, ctas_per_sm=2),
                                    dict(variant=2, ctas_per_sm=1, chunk_batches=1,
                                         rows_per_unit=16),
                                    dict(variant=2, ctas_per_sm=2, chunk_batches=16,
                                         rows_per_unit=1),
                                    dict(queue_order=2, rows_per_unit=1),
                                    dict(queue_order=2, ctas_per_sm=1, rows_per_unit=16),
                                    dict(ctas_per_sm=3),
                                    ],
                         ids=lambda d: ",".join("%s=%d" % kv for kv in d.items()) or "default")
def test_launch_shapes_do_not_change_results(tuning):
    before = _native.get_tuning()
    try:
        _native.set_tuning(**tuning)
        for name, spec in (("decode", wl.SPECS["decode_b256"].with_(B=40)),
                           ("prefill", wl.SPECS["prefill_b8"].with_(
                               B=3, prompt_lo=100, prompt_hi=900, H=256))):
            w = _gen(spec, 7)
            assert_same(run_fused(w), oracle_of(w), what=name)
    finally:
        _native.set_tuning(**before)


# ------------------------------------------------------------------ argmax

def _tie_rows(V, dtype):
    rows = []
    g = torch.Generator().manual_seed(5)

    def base(val=-1.0):
        return torch.full((V,), val)
    r = base(0.0); rows.append(r)                           # all equal -> 0
    r = base(); r[V - 1] = 3; rows.append(r)                # last column
    r = base(); r[0] = 3; r[V - 1] = 3; rows.append(r)      # first and last
    for step in (8, 2048, 8192, 16384, 32768):              # vector / batch edges
        r = base()
        for j in range(step - 1, V, step):
            r[j] = 2
            if j + 1 < V:
                r[j + 1] = 2
        rows.append(r)
    r = base(); r[V // 2 + 1] = 0.0; r[V // 2] = -0.0; rows.append(r)   # -0 first
    r = base(); r[V // 3] = 0.0; r[V // 3 + 1] = -0.0; rows.append(r)   # +0 first
    r = base(-2.0); r[V - 2] = -0.0; r[V - 1] = 0.0; rows.append(r)      # zeros in tail
    for _ in range(6):                                      # random with duplicates
        r = torch.randn(V, generator=g) * 2
        mx = float(r.max()) + 1
        idx = torch.randint(0, V, (5,), generator=g)
        r[idx] = mx
        rows.append(r)
    r = torch.full((V,), float("-inf")); rows.append(r)     # all -inf -> 0
    return torch.stack(rows).to(dtype)


@pytest.mark.parametrize("V,dtype,pad", [(151936, torch.bfloat16, 0),
                                         (201088, torch.bfloat16, 0),
                                         (151937, torch.bfloat16, 7),
                                         (65537, torch.float32, 3),
                                         (1000, torch.float32, 0),
                                         (9, torch.bfloat16, 7)])
@pytest.mark.parametrize("tuning", [dict(), dict(ctas_per_sm=1, chunk_batches=1),
                                    dict(variant=2, ctas_per_sm=1),
                                    dict(variant=2, ctas_per_sm=2, chunk_batches=1)],
                         ids=["default", "coarse", "variant2", "variant2_fine"])
def test_verify_argmax_ties(V, dtype, pad, tuning):
    rows = _tie_rows(V, dtype)
    ref = oracle.argmax_rows(rows)
    import numpy as np
    assert (ref.numpy() == np.argmax(rows.float().numpy(), axis=1)).all()
    base = torch.full((rows.shape[0], V + pad), 100.0, dtype=dtype)  # pad would win
    base[:, :V] = rows
    dev = base.cuda()[:, :V]
    n = rows.shape[0]
    acc = torch.empty(n, dtype=torch.int32, device="cuda")
    bon = torch.empty_like(acc)
    amax = torch.empty_like(acc)
    ws = _native.new_workspace(n, n)
    err = _native.new_error_word()
    before = _native.get_tuning()
    try:
        _native.set_tuning(**tuning)
        _native.verify_greedy(dev, 0, None, acc, bon, ws, err, target_argmax=amax)
    finally:
        _native.set_tuning(**before)
    torch.cuda.synchronize()
    assert torch.equal(amax.cpu(), ref)
    assert torch.equal(bon.cpu(), ref) and (acc.cpu() == 0).all()
    assert int(ws.count_nonzero()) == 0


def test_bonus_equal_to_mask_id():
    w = _gen(wl.SPECS["tiny"].with_(B=6, forced=tuple((b, b % 4) for b in range(6))), 3)
    # make the first mismatching row of every request pick the MASK id
    for b in range(w.B):
        a = int(w.planted_accept[b])
        row = b * (w.Kp + 1) + a
        w.logits[row, w.mask_id] = wl.PLANT * 2
    got = run_fused(w)
    ref = oracle_of(w)
    assert (ref["bonus_token"] == w.mask_id).all()
    assert_same(got, ref, what="bonus=MASK")


# ------------------------------------------------------ separate entry points

@pytest.mark.parametrize("name", ["tiny", "decode_b1", "prefill_small"])
def test_separate_entry_points(name):
    spec = (wl.SPECS[name] if name in wl.SPECS else
            wl.SPECS["prefill_b8"].with_(B=5, prompt_lo=1, prompt_hi=200, V=5003,
                                         row_pad=5, H=72))
    w = _gen(spec, 11)
    wc = w.to("cpu")
    B, Kp, K, R = w.B, w.Kp, w.K, w.R
    # verification
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty_like(acc)
    amax = torch.empty(B * (Kp + 1), dtype=torch.int32, device="cuda")
    ws = _native.new_workspace(B * (Kp + 1), B)
    err = _native.new_error_word()
    _native.verify_greedy(w.logits, Kp, w.in_tokens if Kp else None, acc, bon, ws, err,
                          target_argmax=amax)
    r_acc, r_bon, r_amax = oracle.verify_greedy(wc.logits, B, Kp, w.V, wc.in_tokens)
    torch.cuda.synchronize()
    assert torch.equal(acc.cpu(), r_acc) and torch.equal(bon.cpu(), r_bon)
    assert torch.equal(amax.cpu(), r_amax)
    # rebuild from the verification result
    g = Guarded()
    db = _native.DraftBatch(
        out_offsets=g.alloc((B + 1,), torch.int32), out_tokens=g.alloc((w.T,), torch.int32),
        out_positions=g.alloc((w.T,), torch.int32), is_rejected=g.alloc((w.T,), torch.uint8),
        is_masked=g.alloc((w.T,), torch.uint8), hidden_map=g.alloc((R,), torch.int32),
        slot_mapping=g.alloc((w.T,), torch.int64), sample_idx=g.alloc((B * K,), torch.int32))
    _native.build_draft_batch(B, Kp, K, w.mask_id, R, w.in_offsets, w.in_tokens,
                              w.in_positions, acc, bon, w.block_table, w.block_size, db, err)
    ref, rerr = oracle.build_draft_batch(B, Kp, K, w.mask_id, wc.in_offsets, wc.in_tokens,
                                         wc.in_positions, r_acc, r_bon, wc.block_table,
                                         w.block_size)
    torch.cuda.synchronize()
    g.check()
    for k in ref:
        assert torch.equal(getattr(db, k).cpu(), ref[k].to(getattr(db, k).dtype)), k
    # assembly from the rebuilt batch
    X = g.alloc((w.T, 2 * w.H), w.emb.dtype)
    _native.assemble_draft_inputs(w.emb, w.hidden, w.h_shared, db.out_tokens, db.hidden_map,
                                  db.is_masked, X, err)
    rX, xerr = oracle.assemble_draft_inputs(w.H, w.V, wc.emb, wc.hidden, wc.h_shared,
                                            ref["out_tokens"], ref["hidden_map"],
                                            ref["is_masked"])
    torch.cuda.synchronize()
    g.check()
    assert torch.equal(X.cpu().view(torch.uint8), rX.view(torch.uint8))
    assert int(err.item()) == rerr | xerr == 0
    # and the fused step gives the same as the three calls
    assert_same(run_fused(w), oracle_of(w), what=name + " fused")


def test_assemble_keeps_unmapped_rows_and_skips_bad_map():
    w = _gen(wl.SPECS["tiny"], 2)
    wc = w.to("cpu")
    ref, _ = oracle.build_draft_batch(w.B, w.Kp, w.K, w.mask_id, None, wc.in_tokens,
                                      wc.in_positions, w.planted_accept,
                                      torch.arange(w.B, dtype=torch.int32), wc.block_table, 16)
    hmap = ref["hidden_map"].clone()
    hmap[1] = -4          # out of range: skipped, bit raised
    hmap[2] = w.T + 3     # out of range
    tok = ref["out_tokens"].clone()
    tok[0] = w.V          # out of range: zero embedding half
    X0 = torch.randn(w.T, 2 * w.H)
    rX, rerr = oracle.assemble_draft_inputs(w.H, w.V, wc.emb, wc.hidden, wc.h_shared, tok,
                                            hmap, ref["is_masked"], X=X0)
    X = X0.cuda()
    err = _native.new_error_word()
    _native.assemble_draft_inputs(w.emb, w.hidden, w.h_shared, tok.cuda(), hmap.cuda(),
                                  ref["is_masked"].cuda(), X, err)
    torch.cuda.synchronize()
    assert rerr == oracle.ERR_MAP_RANGE | oracle.ERR_TOKEN_RANGE
    assert int(err.item()) == rerr
    assert torch.equal(X.cpu().view(torch.int32), rX.view(torch.int32))


# ---------------------------------------------------------------- data errors

def test_out_of_range_tokens_and_positions():
    spec = wl.SPECS["tiny"].with_(B=5, forced=((0, 3), (1, 0), (2, 1), (3, 2), (4, 0)))
    w = _gen(spec, 4)
    w.in_tokens[1] = -5            # accepted draft of request 0 (a=3): copied, zero emb
    w.in_tokens[3] = w.V + 3       # last draft of request 0
    w.in_tokens[6] = 2 ** 30       # rejected slot of request 1
    w.in_positions[8:12] = torch.arange(64 * 16 - 2, 64 * 16 + 2, dtype=torch.int32,
                                        device="cuda")   # request 2 runs off the table
    w.in_positions[16] = -7        # request 4's NTP slot: negative position
    got = run_fused(w)
    ref = oracle_of(w)
    assert ref["err"] == oracle.ERR_TOKEN_RANGE | oracle.ERR_BLOCK_RANGE
    assert_same(got, ref, what="data errors")


def test_invalid_prefill_offsets_write_nothing():
    spec = wl.SPECS["prefill_b8"].with_(B=4, prompt_lo=2, prompt_hi=9, V=501, row_pad=3,
                                        H=8)
    w = _gen(spec, 1)
    offs = w.in_offsets.clone()
    offs[2] = offs[1]              # an empty segment
    w.in_offsets = offs
    g = Guarded()
    out = guarded_outputs(w, g)
    ws = _native.new_workspace(w.B, w.B)
    err = _native.new_error_word()
    harness.run(w, out, ws, err)
    torch.cuda.synchronize()
    g.check()
    assert int(err.item()) == _native.ERR_OFFSETS
    assert (out.out_tokens == -123456789).all() and (out.accepted_len == -123456789).all()
    assert int(ws.count_nonzero()) == 0
    ref = oracle_of(w)
    assert ref["err"] == oracle.ERR_OFFSETS


# --------------------------------------------------------------- workspace

def test_workspace_reused_across_calls_and_sizes():
    ws = _native.new_workspace(256 * 8, 256)   # sized for the largest batch
    for i, spec in enumerate([wl.SPECS["decode_b256"].with_(B=256, V=30011, row_pad=5),
                              wl.SPECS["tiny"], wl.SPECS["decode_b256"].with_(B=17),
                              wl.SPECS["prefill_b8"].with_(B=5, prompt_lo=1, prompt_hi=700, H=64),
                              wl.SPECS["decode_b256"].with_(B=256, V=30011, row_pad=5)]):
        w = _gen(spec, 100 + i)
        assert_same(run_fused(w, workspace=ws), oracle_of(w), what="call %d" % i)


def test_back_to_back_calls_without_sync():
    """Several steps queued on one stream share one workspace."""
    ws = _native.new_workspace(64 * 8, 64)
    ws_list = [_gen(wl.SPECS["decode_b64"].with_(B=32, V=50021, row_pad=3), 200 + i)
               for i in range(3)]
    outs = []
    for w in ws_list:
        out, _, err = harness.allocate(w)
        harness.run(w, out, ws, err)
        outs.append((out, err))
    torch.cuda.synchronize()
    for w, (out, err) in zip(ws_list, outs):
        got = harness.to_host(out)
        got["err"] = int(err.item())
        assert_same(got, oracle_of(w))
    assert int(ws.count_nonzero()) == 0


# ------------------------------------------------------------ drafter readout

@pytest.mark.parametrize("variant", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("V,dtype,pad", [(151936, torch.bfloat16, 0), (201088, torch.bfloat16, 0),
                                         (1001, torch.float32, 3), (13, torch.bfloat16, 3)])
def test_draft_readout(V, dtype, pad, variant):
    """Greedy t_1..t_K: the drafter's logits over all output slots, read
    through the sample_idx the rebuild wrote; and over the sampled rows only."""
    w = _gen(wl.SPECS["decode_b256"].with_(B=24, V=V, row_pad=pad, H=64, dtype=dtype), 3)
    out, ws, err = harness.allocate(w)
    harness.run(w, out, ws, err)
    g = torch.Generator(device="cuda").manual_seed(9)
    T = w.T
    base = torch.randint(-3, 4, (T, V + pad), generator=g, device="cuda").to(dtype)
    drafter = base[:, :V]                           # ties everywhere
    sidx = out.sample_idx
    tok = torch.full((sidx.numel(),), -9, dtype=torch.int32, device="cuda")
    rws = _native.new_workspace(sidx.numel(), sidx.numel())
    rerr = _native.new_error_word()
    with tuned(**variant):
        _native.draft_readout(drafter, tok, rws, rerr, sample_idx=sidx)
        only = base[sidx.long()][:, :V]             # [B*K, V] rows, padded stride
        tok2 = torch.full_like(tok, -9)
        _native.draft_readout(only, tok2, rws, rerr)
    torch.cuda.synchronize()
    ref, e = oracle.draft_readout(drafter.cpu(), sidx.cpu())
    assert e == 0 and int(rerr.item()) == 0
    assert torch.equal(tok.cpu(), ref) and torch.equal(tok2.cpu(), ref)
    assert int(rws.count_nonzero()) == 0


def test_draft_readout_bad_rows():
    logits = torch.randn(40, 1000, device="cuda")
    idx = torch.tensor([5, -1, 40, 39, 2 ** 30], dtype=torch.int32, device="cuda")
    tok = torch.full((5,), -9, dtype=torch.int32, device="cuda")
    ws = _native.new_workspace(5, 5)
    err = _native.new_error_word()
    _native.draft_readout(logits, tok, ws, err, sample_idx=idx)
    torch.cuda.synchronize()
    ref, e = oracle.draft_readout(logits.cpu(), idx.cpu())
    assert e == oracle.ERR_ROW_RANGE == int(err.item())
    assert torch.equal(tok.cpu(), ref)
    assert int(ws.count_nonzero()) == 0
