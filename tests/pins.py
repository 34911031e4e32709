"""Checks that pin the CPU oracle to facts fixed outside of it.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something the pages or plain mathematics fix: a brute-force enumeration, a
library routine with a documented tie rule (numpy / torch argmax, torch
indexing), an invariant that holds by construction of the inputs (planted
acceptance lengths), or a hand-worked example under ``tests/golden``.
``test_oracle_pins.py`` runs them against the oracle; ``test_oracle_mutants.py``
runs them against deliberately broken copies of the oracle to show that each
plausible mistake is caught.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch

import oracle
from speculative_decoding_pe_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- argmax (a1)

def pin_argmax_bruteforce():
    """All rows over {-1, -0, +0, 1, 2}^V for V <= 5, both dtypes: the answer
    is the first index whose value equals the row maximum (numeric compare,
    so -0.0 == +0.0)."""
    alphabet = [-1.0, -0.0, 0.0, 1.0, 2.0]
    for V in range(1, 6):
        rows = list(itertools.product(alphabet, repeat=V))
        expect = []
        for r in rows:
            mx = max(r)
            expect.append(next(i for i, x in enumerate(r) if x == mx))
        for dt in (torch.float32, torch.bfloat16):
            t = torch.tensor(rows, dtype=dt)
            got = oracle.argmax_rows(t).tolist()
            assert got == expect, "argmax brute force V=%d %s" % (V, dt)


def pin_argmax_numpy():
    """numpy.argmax documents that the first occurrence of the maximum wins;
    draw rows from a few values so that ties are everywhere, plus normal
    rows, fp32 and bf16, with a padded row stride."""
    g = torch.Generator().manual_seed(11)
    for dt in (torch.float32, torch.bfloat16):
        for V in (1, 7, 33, 1000, 4099):
            few = torch.randint(-3, 3, (40, V), generator=g).to(dt)
            nrm = torch.randn(40, V, generator=g).to(dt)
            for t in (few, nrm):
                ref = np.argmax(t.float().numpy(), axis=1)
                assert (oracle.argmax_rows(t).numpy() == ref).all()
                pad = torch.full((40, V + 5), 1e30).to(dt)
                pad[:, :V] = t
                got = oracle.argmax_rows(pad[:, :V], V).numpy()
                assert (got == ref).all(), "row stride ignored"


def pin_draft_readout():
    """Greedy draft tokens are numpy.argmax (first occurrence) of the rows the
    drafter's LM head reads; an index outside the logits gives -1."""
    g = torch.Generator().manual_seed(23)
    for dt in (torch.float32, torch.bfloat16):
        logits = torch.randint(-2, 3, (50, 777), generator=g).to(dt)
        idx = torch.randint(0, 50, (64,), generator=g, dtype=torch.int32)
        got, err = oracle.draft_readout(logits, idx)
        ref = np.argmax(logits.float().numpy(), axis=1)[idx.numpy()]
        assert err == 0 and (got.numpy() == ref).all()
        got, err = oracle.draft_readout(logits)          # identity rows
        assert err == 0 and (got.numpy() == np.argmax(logits.float().numpy(), axis=1)).all()
        bad = torch.tensor([3, -1, 50, 7], dtype=torch.int32)
        got, err = oracle.draft_readout(logits, bad)
        assert err == oracle.ERR_ROW_RANGE
        assert got[1] == -1 and got[2] == -1
        assert got[0] == int(np.argmax(logits[3].float().numpy()))


# ----------------------------------------------------------- acceptance (a2)

def pin_accept_enumeration():
    """V=3, K'=3: every draft sequence (3^3) x every target-argmax sequence
    (3^4).  Accepted length counted as the number of leading drafts whose
    whole prefix matches; bonus is the target choice right after them."""
    V, Kp = 3, 3
    cases = [(d, g) for d in itertools.product(range(V), repeat=Kp)
             for g in itertools.product(range(V), repeat=Kp + 1)]
    B = len(cases)
    logits = torch.zeros(B * (Kp + 1), V)
    tokens = torch.zeros(B * (Kp + 1), dtype=torch.int32)
    exp_a, exp_bonus = [], []
    for b, (d, g) in enumerate(cases):
        for j in range(Kp + 1):
            logits[b * (Kp + 1) + j, g[j]] = 1.0
        tokens[b * (Kp + 1)] = 0
        tokens[b * (Kp + 1) + 1: (b + 1) * (Kp + 1)] = torch.tensor(d)
        a = sum(1 for j in range(Kp) if all(d[i] == g[i] for i in range(j + 1)))
        exp_a.append(a)
        exp_bonus.append(g[a])
    acc, bon, amax = oracle.verify_greedy(logits, B, Kp, V, tokens)
    assert acc.tolist() == exp_a
    assert bon.tolist() == exp_bonus


def pin_planted(spec_names=("tiny",), seeds=(0, 1, 2, 3)):
    """The generator plants a unique row maximum on each row of the accepted
    prefix (equal to the draft) and on the first mismatching row (not equal
    to the draft): any greedy verifier must return the planted length, and
    the planted column as bonus."""
    for name in spec_names:
        for seed in seeds:
            w = wl.make_workload(name, seed)
            acc, bon, _ = oracle.verify_greedy(w.logits, w.B, w.Kp, w.V, w.in_tokens)
            assert torch.equal(acc, w.planted_accept), (name, seed)
            known = w.planted_bonus >= 0
            assert torch.equal(bon[known], w.planted_bonus[known]), (name, seed)


# ------------------------------------------------ rejection sampling (next row)

def pin_philox_known_answers():
    """Philox4x32-10 reproduces the known-answer vectors published with the
    generator (Salmon et al., SC'11; Random123 distribution)."""
    kat = [((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
           ((0xffffffff,) * 4, (0xffffffff,) * 2,
            (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
           ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
            (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1))]
    for ctr, key, want in kat:
        assert tuple(oracle.philox4x32_10(ctr, key)) == want


def _sharp_case(B=40, Kp=5, V=61, seed=3):
    """Target rows with distinct integer logits and draft rows one-hot at the
    draft token; planted acceptance as in the synthetic workloads."""
    g = torch.Generator().manual_seed(seed)
    t = torch.stack([torch.randperm(V, generator=g).float() for _ in range(B * (Kp + 1))])
    amax = t.argmax(1)
    tokens = torch.randint(0, V, (B * (Kp + 1),), generator=g, dtype=torch.int32)
    for b in range(B):
        a = int(torch.randint(0, Kp + 1, (), generator=g))
        for j in range(Kp):
            row = b * (Kp + 1) + j
            if j < a:
                tokens[row + 1] = amax[row]
            elif j == a and int(tokens[row + 1]) == int(amax[row]):
                tokens[row + 1] = (amax[row] + 1) % V
    d = torch.full((B * Kp, V), -50.0)
    for b in range(B):
        for j in range(Kp):
            d[b * Kp + j, int(tokens[b * (Kp + 1) + j + 1])] = 50.0
    u = torch.rand(B * Kp, generator=g) * 0.999 + 0.0005
    return t, d, tokens, u


def pin_sampled_cold_is_greedy():
    """At a cold temperature with one-hot drafts, speculative sampling must
    accept exactly the drafts greedy verification accepts and draw the
    greedy bonus (the target's distribution is then one-hot)."""
    B, Kp = 40, 5
    t, d, tokens, u = _sharp_case(B, Kp)
    acc, bon = oracle.verify_sampled(t, d, B, Kp, tokens, u, 0.01, 11)
    gacc, gbon, _ = oracle.verify_greedy(t, B, Kp, t.shape[1], tokens)
    assert torch.equal(acc, gacc) and torch.equal(bon, gbon)
    assert 0 < int((acc == Kp).sum()) < B and int((acc < Kp).sum()) > 0


def pin_sampled_same_distribution_accepts_all():
    """When the drafter's distribution equals the target's, every draft is
    accepted (u * q(x) < p(x) for every u in [0, 1))."""
    g = torch.Generator().manual_seed(5)
    B, Kp, V = 30, 4, 97
    t = torch.randn(B * (Kp + 1), V, generator=g)
    d = torch.stack([t[b * (Kp + 1) + j] for b in range(B) for j in range(Kp)])
    tokens = torch.randint(0, V, (B * (Kp + 1),), generator=g, dtype=torch.int32)
    u = torch.rand(B * Kp, generator=g)
    acc, _ = oracle.verify_sampled(t, d, B, Kp, tokens, u, 0.7, 3)
    assert (acc == Kp).all()


def _chi2(counts, probs):
    n = counts.sum()
    exp = probs * n
    return float(((counts - exp) ** 2 / exp).sum())


def pin_sampled_preserves_target_distribution():
    """The guarantee of speculative sampling: whatever the drafter proposes,
    the first emitted token is distributed as the target's p_0, and after an
    accepted draft the bonus is distributed as p_1 (chi-square, 3 degrees of
    freedom, 99.9 % quantile 16.27, over 40000 draws)."""
    rng = np.random.default_rng(17)
    N, V = 40000, 4
    p0 = np.array([0.1, 0.2, 0.3, 0.4])
    p1 = np.array([0.4, 0.3, 0.2, 0.1])
    q0 = np.array([0.4, 0.4, 0.1, 0.1])
    t = torch.tensor(np.log(np.stack([p0, p1] * N)), dtype=torch.float32)
    d = torch.tensor(np.log(np.stack([q0] * N)), dtype=torch.float32)
    x = rng.choice(V, size=N, p=q0)
    tokens = torch.zeros(2 * N, dtype=torch.int32)
    tokens[1::2] = torch.tensor(x, dtype=torch.int32)
    u = torch.tensor(rng.random(N), dtype=torch.float32)
    acc, bon = oracle.verify_sampled(t, d, N, 1, tokens, u, 1.0, 2024)
    acc, bon = acc.numpy(), bon.numpy()
    assert ((acc >= 0) & (acc <= 1)).all() and ((bon >= 0) & (bon < V)).all()
    first = np.where(acc >= 1, x, bon)
    assert _chi2(np.bincount(first, minlength=V), p0) < 16.27
    after = bon[acc == 1]
    assert _chi2(np.bincount(after, minlength=V), p1) < 16.27
    # a plain draw (no drafts) is distributed as p_0 too
    acc0, bon0 = oracle.verify_sampled(t[0::2].contiguous(), None, N, 0, None, None, 1.0, 99)
    assert ((bon0 >= 0) & (bon0 < V)).all()
    assert _chi2(np.bincount(bon0.numpy(), minlength=V), p0) < 16.27


def pin_sampled_residual_across_chunks():
    """The same guarantee on a wide row whose support is four far-apart
    columns (0, 2048, 1, 2049: the residual weight 0.2 and 0.3 sits in
    columns 1 and 2049, the other two cancel), so that any per-chunk or
    per-column bookkeeping of the draw is exercised: the first emitted
    token must follow p_0 over those columns (chi-square, 3 degrees of
    freedom, 99.9 % quantile 16.27, over 4000 requests)."""
    rng = np.random.default_rng(29)
    N, V = 4000, 4096
    cols = np.array([0, 2048, 1, 2049])  # entries of p0 / q0 -> columns
    p0 = np.array([0.1, 0.2, 0.3, 0.4])
    p1 = np.array([0.4, 0.3, 0.2, 0.1])
    q0 = np.array([0.4, 0.4, 0.1, 0.1])
    t = torch.full((2 * N, V), -1.0e4, dtype=torch.float32)
    t[0::2, cols] = torch.tensor(np.log(p0), dtype=torch.float32)
    t[1::2, cols] = torch.tensor(np.log(p1), dtype=torch.float32)
    d = torch.full((N, V), -1.0e4, dtype=torch.float32)
    d[:, cols] = torch.tensor(np.log(q0), dtype=torch.float32)
    x = cols[rng.choice(4, size=N, p=q0)]
    tokens = torch.zeros(2 * N, dtype=torch.int32)
    tokens[1::2] = torch.tensor(x, dtype=torch.int32)
    u = torch.tensor(rng.random(N), dtype=torch.float32)
    acc, bon = oracle.verify_sampled(t, d, N, 1, tokens, u, 1.0, 31)
    acc, bon = acc.numpy(), bon.numpy()
    first = np.where(acc >= 1, x, bon)
    assert np.isin(first, cols).all()
    counts = np.array([(first == c).sum() for c in cols])
    assert _chi2(counts, p0) < 16.27


# -------------------------------------------------- rebuild invariants (a3-a5)

def check_rebuild_invariants(w, o):
    """Closed-form facts about one rebuilt batch (decode or prefill)."""
    B, Kp, K, bs = w.B, w.Kp, w.K, w.block_size
    io = (w.in_offsets.tolist() if w.in_offsets is not None
          else [b * (Kp + 1) for b in range(B + 1)])
    oo = o["out_offsets"].tolist()
    acc = o["accepted_len"].tolist() if "accepted_len" in o else [0] * B
    tok_out, pos_out = o["out_tokens"], o["out_positions"]
    rej, msk = o["is_rejected"].long(), o["is_masked"].long()
    slot, hmap = o["slot_mapping"], o["hidden_map"]
    T = w.R + B * (K - 1)
    assert oo[0] == 0 and oo[B] == T
    assert int(msk.sum()) == B * (K - 1), "one MASK slot per extra draft"
    bt = w.block_table.long()
    used = set()
    exp_rej = 0
    for b in range(B):
        n = io[b + 1] - io[b]
        assert oo[b + 1] - oo[b] == n + K - 1, "rows per request"
        s = n - 1 - Kp + acc[b]
        exp_rej += n - 1 - s
        seg = slice(oo[b], oo[b + 1])
        # the bonus sits at the NTP slot; nothing before it is rejected
        assert int(tok_out[oo[b] + s]) == int(o["bonus_token"][b])
        assert rej[seg].tolist() == [0] * (s + 1) + [1] * (n - 1 - s) + [0] * (K - 1)
        assert msk[seg].tolist() == [0] * n + [1] * (K - 1)
        # positions of the kept slots run on from the first position
        kept = [int(pos_out[t]) for t in range(oo[b], oo[b + 1]) if not rej[t]]
        p0 = int(w.in_positions[io[b]])
        assert kept == list(range(p0, p0 + s + K)), "kept positions contiguous"
        # hidden rows keep their order inside the segment
        assert hmap[io[b]:io[b + 1]].tolist() == list(range(oo[b], oo[b] + n))
        # the drafter reads the NTP slot, then the MASK slots
        sidx = o["sample_idx"][b * K:(b + 1) * K].tolist()
        assert sidx == [oo[b] + s] + [t for t in range(oo[b], oo[b + 1]) if msk[t]]
        # paged KV: rejected slots padded, others inside the request's blocks
        row = set(bt[b].tolist())
        for t in range(oo[b], oo[b + 1]):
            sl, p = int(slot[t]), int(pos_out[t])
            if rej[t]:
                assert sl == -1, "rejected slot must be padded"
            else:
                assert sl >= 0 and sl % bs == p % bs and (sl // bs) in row
                assert sl not in used or w.spec.bt_per_row
                used.add(sl)
        # consecutive kept positions in one block -> consecutive slots
        kept_t = [t for t in range(oo[b], oo[b + 1]) if not rej[t]]
        for t0, t1 in zip(kept_t, kept_t[1:]):
            p_a, p_b = int(pos_out[t0]), int(pos_out[t1])
            if p_b == p_a + 1 and p_a // bs == p_b // bs:
                assert int(slot[t1]) == int(slot[t0]) + 1
    assert int(rej.sum()) == exp_rej


def check_prefill_shift(w, o):
    """Prompt slot k pairs token k+1 with hidden row k (shift by one)."""
    io = w.in_offsets.tolist()
    for b in range(w.B):
        n = io[b + 1] - io[b]
        oo = int(o["out_offsets"][b])
        got = o["out_tokens"][oo:oo + n - 1]
        assert torch.equal(got, w.in_tokens[io[b] + 1:io[b + 1]])


def check_assembly(w, o):
    """X against independent torch statements: the embedding half is an
    index_select of the table; the hidden half is a scatter of the target
    rows through the hidden-state mapping followed by a masked overwrite with
    h_shared; every MASK row is emb(mask) (+) h_shared."""
    H = w.H
    X = o["X"]
    tok = o["out_tokens"].long()
    assert torch.equal(X[:, :H], torch.index_select(w.emb.cpu(), 0, tok))
    hs = torch.zeros(X.shape[0], H, dtype=X.dtype)
    hs[o["hidden_map"].long()] = w.hidden.cpu()
    msk = o["is_masked"].bool()
    hs = torch.where(msk.unsqueeze(1), w.h_shared.cpu(), hs)
    assert torch.equal(X[:, H:], hs)
    mask_row = torch.cat([w.emb[w.mask_id].cpu(), w.h_shared.cpu()])
    assert torch.equal(X[msk], mask_row.expand(int(msk.sum()), -1))


def _small_specs():
    base = wl.SPECS["tiny"]
    return [
        base,
        base.with_(name="tiny_bf16", dtype=torch.bfloat16, B=9, Kp=5, K=4),
        base.with_(name="k1", K=1, B=5),
        base.with_(name="kp1", Kp=1, K=6, B=6, accept_p=0.5),
        base.with_(name="all_none", B=2, Kp=4, K=2, forced=((0, 4), (1, 0))),
        base.with_(name="global_bt", B=7, bt_per_row=False, bt_width=40),
        base.with_(name="prefill", Kp=0, K=4, B=5, prompt_lo=1, prompt_hi=40,
                   bt_width=4, bt_per_row=False, V=777, row_pad=3),
        base.with_(name="prefill_k1", Kp=0, K=1, B=3, prompt_lo=1, prompt_hi=9,
                   bt_width=2),
        base.with_(name="b1", B=1, Kp=7, K=7, V=513, row_pad=3),
    ]


def pin_step_invariants(seeds=(0, 1)):
    for spec in _small_specs():
        for seed in seeds:
            w = wl.make_workload(spec, seed)
            o = oracle.step(w)
            assert o["err"] == 0, (spec.name, o["err"])
            if not spec.prefill:
                assert torch.equal(o["accepted_len"], w.planted_accept), spec.name
            else:
                assert (o["accepted_len"] == 0).all()
                check_prefill_shift(w, o)
            check_rebuild_invariants(w, o)
            check_assembly(w, o)
            ref = np.argmax(w.logits.float().numpy(), axis=1)
            assert (o["target_argmax"].numpy() == ref).all()


# ------------------------------------------------------------ golden examples

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _identifiable_tables(V, H, R):
    """Embedding row v = (v, 100+v), hidden row i = (1000+i, 2000+i),
    h_shared = (-5, -6): every X row names its own sources."""
    emb = torch.tensor([[v, 100 + v] for v in range(V)], dtype=torch.float32)
    hid = torch.tensor([[1000 + i, 2000 + i] for i in range(R)], dtype=torch.float32)
    hs = torch.tensor([-5.0, -6.0])
    return emb, hid, hs


def _x_expect(rows, emb, hid, hs):
    out = []
    for r in rows:
        e = emb[r[1]]
        h = hs if r[2] == "shared" else hid[r[3]]
        out.append(torch.cat([e, h]))
    return torch.stack(out)


class _W:
    """Minimal workload record for golden examples."""
    def __init__(self, **kw):
        self.__dict__.update(kw)


def pin_golden_decode():
    g = _golden("decode_worked_example.json")
    B, Kp, K, V, H = g["B"], g["Kp"], g["K"], g["V"], g["H"]
    logits = torch.full((B * (Kp + 1), V), g["logits_base"])
    for r, sets in enumerate(g["logits_rows"]):
        for c, v in sets.items():
            logits[r, int(c)] = v
    R = B * (Kp + 1)
    emb, hid, hs = _identifiable_tables(V, H, R)
    w = _W(B=B, Kp=Kp, K=K, V=V, H=H, mask_id=g["mask_id"],
           block_size=g["block_size"], logits=logits, in_offsets=None,
           in_tokens=torch.tensor(g["in_tokens"], dtype=torch.int32),
           in_positions=torch.tensor(g["in_positions"], dtype=torch.int32),
           block_table=torch.tensor(g["block_table"], dtype=torch.int32),
           emb=emb, hidden=hid, h_shared=hs)
    o = oracle.step(w)
    e = g["expect"]
    assert o["err"] == 0
    for key in ("target_argmax", "accepted_len", "bonus_token", "out_offsets",
                "out_tokens", "out_positions", "is_rejected", "is_masked",
                "slot_mapping", "hidden_map", "sample_idx"):
        assert o[key].tolist() == e[key], key
    assert torch.equal(o["X"], _x_expect(e["x_rows"], emb, hid, hs))


def pin_golden_prefill():
    g = _golden("prefill_input_rule.json")
    B, K, V, H = g["B"], g["K"], g["V"], g["H"]
    L = len(g["prompt_tokens"])
    logits = torch.full((1, V), g["last_row_logits"]["base"])
    for c, v in g["last_row_logits"]["set"].items():
        logits[0, int(c)] = v
    emb, hid, hs = _identifiable_tables(V, H, L)
    w = _W(B=B, Kp=0, K=K, V=V, H=H, mask_id=g["mask_id"],
           block_size=g["block_size"], logits=logits,
           in_offsets=torch.tensor([0, L], dtype=torch.int32),
           in_tokens=torch.tensor(g["prompt_tokens"], dtype=torch.int32),
           in_positions=torch.arange(L, dtype=torch.int32),
           block_table=torch.tensor(g["block_table"], dtype=torch.int32),
           emb=emb, hidden=hid, h_shared=hs)
    o = oracle.step(w)
    e = g["expect"]
    assert o["err"] == 0
    assert o["bonus_token"].tolist() == [e["new_token"]]
    for key in ("out_tokens", "out_positions", "is_rejected", "is_masked",
                "slot_mapping", "sample_idx"):
        assert o[key].tolist() == e[key], key
    assert torch.equal(o["X"], _x_expect(e["x_rows"], emb, hid, hs))


# ----------------------------------------------------------- data-error rules

def pin_error_rules():
    """Out-of-range data never reads or writes outside a buffer: a token
    outside [0,V) gathers a zero row, a position outside the block table gets
    slot -1, a bad accepted length counts as 0; each raises its bit."""
    w = wl.make_workload(wl.SPECS["tiny"].with_(B=3), 5)
    acc = torch.tensor([1, 9, -1], dtype=torch.int32)   # 9 > Kp, -1 < 0
    bonus = torch.tensor([7, 8, 9], dtype=torch.int32)
    pos = w.in_positions.clone()
    pos[4] = -3                                           # request 1, slot 0
    pos[8] = 64 * 16 + 5                                  # past the table
    o, err = oracle.build_draft_batch(w.B, w.Kp, w.K, w.mask_id, None, w.in_tokens,
                                      pos, acc, bonus, w.block_table, 16)
    assert err == oracle.ERR_SLOT_RANGE | oracle.ERR_BLOCK_RANGE
    m = w.Kp + w.K
    assert int(o["out_tokens"][m + 0]) == 8               # a=9 treated as 0
    assert int(o["out_tokens"][2 * m + 0]) == 9           # a=-1 treated as 0
    assert int(o["slot_mapping"][m + 0]) == -1
    assert int(o["slot_mapping"][2 * m + 0]) == -1
    tok = o["out_tokens"].clone()
    tok[0], tok[1] = -1, w.V
    X, err = oracle.assemble_draft_inputs(w.H, w.V, w.emb, w.hidden, w.h_shared, tok,
                                          o["hidden_map"], o["is_masked"])
    assert err == oracle.ERR_TOKEN_RANGE
    assert (X[0, :w.H] == 0).all() and (X[1, :w.H] == 0).all()
    hmap = o["hidden_map"].clone()
    hmap[0] = -2
    X2, err = oracle.assemble_draft_inputs(w.H, w.V, w.emb, w.hidden, w.h_shared,
                                           o["out_tokens"], hmap, o["is_masked"])
    assert err == oracle.ERR_MAP_RANGE
    # bad prefill offsets: nothing written
    offs = torch.tensor([0, 3, 3, 5], dtype=torch.int32)  # empty segment
    o3, err = oracle.build_draft_batch(3, 0, 2, w.mask_id, offs, w.in_tokens[:5],
                                       w.in_positions[:5], None, bonus,
                                       w.block_table, 16)
    assert err == oracle.ERR_OFFSETS
    assert (o3["out_tokens"] == -7).all()


ALL_PINS = [pin_argmax_bruteforce, pin_argmax_numpy, pin_draft_readout,
            pin_philox_known_answers, pin_sampled_cold_is_greedy,
            pin_sampled_same_distribution_accepts_all,
            pin_sampled_preserves_target_distribution, pin_sampled_residual_across_chunks,
            pin_accept_enumeration,
            pin_planted, pin_step_invariants, pin_golden_decode,
            pin_golden_prefill, pin_error_rules]
