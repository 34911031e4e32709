"""Helpers for the GPU parity tests: guard-banded outputs and oracle runs."""
from __future__ import annotations

import torch

import oracle
from speculative_decoding_pe_gb300 import _native, harness

GUARD = 64  # elements on each side; keeps 16-byte alignment for every dtype
_SENTINEL = {torch.int32: -123456789, torch.int64: -987654321, torch.uint8: 0xA5}


class Guarded:
    """Buffers that sit between two guard bands filled with a sentinel, and are
    themselves pre-filled with it, so stray and missing writes both show."""

    def __init__(self):
        self.bases = []

    def alloc(self, shape, dtype, device="cuda"):
        n = 1
        for s in shape:
            n *= s
        base = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        if dtype in _SENTINEL:
            base.fill_(_SENTINEL[dtype])
        else:  # floating: a NaN bit pattern
            base.view(torch.uint8).fill_(0xFF)
        view = base[GUARD:GUARD + n].view(*shape)
        self.bases.append((base, n))
        return view

    def check(self):
        for base, n in self.bases:
            esz = base.element_size()
            raw = base.view(torch.uint8)
            if base.dtype in _SENTINEL:
                want = torch.full((GUARD,), _SENTINEL[base.dtype], dtype=base.dtype,
                                  device=base.device).view(torch.uint8)
            else:
                want = torch.full((GUARD * esz,), 0xFF, dtype=torch.uint8,
                                  device=base.device)
            assert torch.equal(raw[:GUARD * esz], want), "write below a buffer"
            assert torch.equal(raw[(GUARD + n) * esz:], want), "write past a buffer"


def guarded_outputs(w, g: Guarded, sample_idx=True, target_argmax=True):
    B, Kp, K, R, H = w.B, w.Kp, w.K, w.R, w.H
    T = R + B * (K - 1)
    return _native.StepOutputs(
        out_offsets=g.alloc((B + 1,), torch.int32),
        out_tokens=g.alloc((T,), torch.int32),
        out_positions=g.alloc((T,), torch.int32),
        is_rejected=g.alloc((T,), torch.uint8),
        is_masked=g.alloc((T,), torch.uint8),
        hidden_map=g.alloc((R,), torch.int32),
        slot_mapping=g.alloc((T,), torch.int64),
        sample_idx=g.alloc((B * K,), torch.int32) if sample_idx else None,
        accepted_len=g.alloc((B,), torch.int32),
        bonus_token=g.alloc((B,), torch.int32),
        target_argmax=g.alloc((B * (Kp + 1),), torch.int32) if target_argmax else None,
        X=g.alloc((T, 2 * H), w.emb.dtype))


def run_fused(w, workspace=None, check_ws_zero=True):
    """pe_step on GPU workload ``w``; returns host outputs and the error word."""
    g = Guarded()
    out = guarded_outputs(w, g)
    ws = workspace if workspace is not None else _native.new_workspace(
        w.B * (w.Kp + 1), w.B)
    err = _native.new_error_word()
    harness.run(w, out, ws, err)
    torch.cuda.synchronize()
    g.check()
    if check_ws_zero:
        assert int(ws.count_nonzero()) == 0, "workspace not left zeroed"
    res = harness.to_host(out)
    res["err"] = int(err.item())
    return res


def oracle_of(w) -> dict:
    return oracle.step(w.to("cpu"))


def assert_same(got: dict, ref: dict, keys=None, what=""):
    keys = keys or [k for k in harness.OUTPUT_KEYS if k in got] + ["err"]
    for k in keys:
        a, b = got[k], ref[k]
        if k == "err":
            assert a == b, "%s err word %d != oracle %d" % (what, a, b)
            continue
        if k == "X":  # bit patterns: catches -0.0 vs +0.0 and NaN leftovers
            a = a.contiguous().view(torch.uint8).view(a.shape[0], -1)
            b = b.contiguous().view(torch.uint8).view(b.shape[0], -1)
            same = torch.equal(a, b)
        else:
            same = torch.equal(a, b.to(a.dtype))
        if not same:
            if a.dim() == 2:
                bad = (a != b).any(dim=1).nonzero().flatten()[:5].tolist()
            else:
                bad = (a != b.to(a.dtype)).nonzero().flatten()[:5].tolist()
            first = bad[:1]
            raise AssertionError("%s %s differs from the oracle at %s: got %s want %s" % (
                what, k, bad, a[first].tolist(), b[first].tolist()))
