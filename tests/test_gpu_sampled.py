"""Rejection-sampling verification (pe_verify_sampled) against the CPU oracle.

The kernel decides in fp32 and the oracle in fp64, so a decision may differ
only where the exact quantity is within rounding of the threshold: an accept
test whose p(x) - u q(x) is a tiny fraction of p(x), or a draw whose two best
Gumbel scores are nearly equal.  Every difference is explained that way
(``_explain``) and at most one request in 200 may need it; everything else is
equal element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_util import Guarded
from speculative_decoding_pe_gb300 import _native, build
from speculative_decoding_pe_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ACCEPT_REL_TOL = 1e-4   # |p - u q| / p below which fp32 and fp64 may disagree
SCORE_TOL = 1e-3        # Gumbel score gap below which draws may disagree


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


def run_gpu(s, T, seed, workspace=None, check_ws_zero=True):
    """pe_verify_sampled on inputs ``s`` (moved to the GPU); host outputs."""
    d = s.to("cuda")
    g = Guarded()
    acc = g.alloc((s.B,), torch.int32)
    bon = g.alloc((s.B,), torch.int32)
    ws = workspace if workspace is not None else torch.zeros(
        _native.workspace_bytes_sampled(s.B, s.Kp), dtype=torch.uint8, device="cuda")
    err = _native.new_error_word()
    _native.verify_sampled(d.target_logits, d.draft_logits if s.Kp else None, s.Kp,
                           d.tokens if s.Kp else None, d.u_accept if s.Kp else None,
                           T, seed, acc, bon, ws, err)
    torch.cuda.synchronize()
    g.check()
    if check_ws_zero:
        assert int(ws.count_nonzero()) == 0, "workspace not left zeroed"
    assert int(err.item()) == 0
    return acc.cpu(), bon.cpu()


def run_oracle(s, T, seed):
    return oracle.verify_sampled(s.target_logits, s.draft_logits if s.Kp else None, s.B,
                                 s.Kp, s.tokens if s.Kp else None,
                                 s.u_accept if s.Kp else None, T, seed)


# ------------------------------------------------- exact evaluation of margins

def _gumbel(seed, b, v):
    w = oracle.philox4x32_10((v // 4, b, 0, 0), (seed & 0xFFFFFFFF, seed >> 32))[v % 4]
    u = ((w >> 9) + 0.5) / 8388608.0
    return -math.log(-math.log(u))


def _probs(row, T):
    z = row.double() / T
    return torch.softmax(z, 0)


def _explain(s, T, seed, b, got, ref):
    """Why request b's fp32 result (got) may differ from the fp64 one (ref)."""
    Kp = s.Kp
    ga, gb = got
    ra, rb = ref
    if ga != ra:
        j = min(ga, ra)
        x = int(s.tokens[b * (Kp + 1) + j + 1])
        p = float(_probs(s.target_logits[b * (Kp + 1) + j], T)[x])
        q = float(_probs(s.draft_logits[b * Kp + j], T)[x])
        u = float(s.u_accept[b * Kp + j])
        margin = abs(p - u * q) / max(p, 1e-300)
        assert margin < ACCEPT_REL_TOL, (
            "request %d: accepted %d, oracle %d; p(x)=%g u q(x)=%g is no near tie" % (
                b, ga, ra, p, u * q))
        return
    a = ra
    p = _probs(s.target_logits[b * (Kp + 1) + a], T)
    if a < Kp:
        q = _probs(s.draft_logits[b * Kp + a], T)
        r = torch.clamp(p - q, min=0)
        w = r if float(r.sum()) > 0 else p
    else:
        w = p

    def score(v):
        return math.log(float(w[v])) + _gumbel(seed, b, v) if float(w[v]) > 0 else -math.inf

    sg, sr = score(gb), score(rb)
    assert abs(sg - sr) < SCORE_TOL, (
        "request %d: bonus %d (score %g), oracle %d (score %g): no near tie" % (
            b, gb, sg, rb, sr))


def assert_parity(s, T, seed, got, ref):
    acc, bon = got
    racc, rbon = ref
    diff = ((acc != racc) | (bon != rbon)).nonzero().flatten().tolist()
    for b in diff:
        _explain(s, T, seed, b, (int(acc[b]), int(bon[b])), (int(racc[b]), int(rbon[b])))
    assert len(diff) <= max(1, s.B // 200), "%d requests differ: %s" % (len(diff), diff[:8])
    assert ((acc >= 0) & (acc <= s.Kp)).all()
    assert ((bon >= 0) & (bon < s.V)).all()


CASES = [
    # name, B, Kp, V, dtype, temperature, seed
    ("tiny_f32_tail", 5, 3, 37, torch.float32, 1.0, 1),
    ("V_below_one_vector", 4, 2, 5, torch.bfloat16, 1.0, 2),
    ("bf16_ragged", 7, 4, 1003, torch.bfloat16, 0.8, 3),
    ("many_chunks_ragged", 3, 2, 70001, torch.bfloat16, 1.3, 4),
    ("first_draft_after_prefill_Kp0", 16, 0, 32000, torch.bfloat16, 1.0, 5),
    ("many_small_rows", 1000, 1, 64, torch.float32, 0.9, 6),
    ("f32_mid", 32, 7, 50000, torch.float32, 0.6, 7),
    ("cold_T0.25", 64, 7, 32000, torch.bfloat16, 0.25, 10),
    ("hot_T4_f32", 48, 5, 32003, torch.float32, 4.0, 11),
    ("decode_b64_V201088", 64, 7, 201088, torch.bfloat16, 1.0, 8),
    ("decode_b256_V151936", 256, 7, 151936, torch.bfloat16, 1.0, 9),
]


@pytest.mark.parametrize("name,B,Kp,V,dtype,T,seed", CASES, ids=[c[0] for c in CASES])
def test_sampled_parity(name, B, Kp, V, dtype, T, seed):
    s = wl.make_sampled_inputs(B, Kp, V, dtype=dtype, seed=seed)
    ref = run_oracle(s, T, 1000 + seed)
    got = run_gpu(s, T, 1000 + seed)
    assert_parity(s, T, 1000 + seed, got, ref)
    if Kp and B >= 8:  # the inputs mix fully accepted requests with rejections
        assert 0 < int((ref[0] == Kp).sum()) < B


def test_sampled_invalid_draft_tokens_are_rejected():
    s = wl.make_sampled_inputs(24, 5, 3001, dtype=torch.bfloat16, seed=11)
    for b in range(24):  # tokens -1 and V at a few positions
        if b % 3 == 0:
            s.tokens[b * 6 + 1 + b % 5] = -1 if b % 2 else 3001
    ref = run_oracle(s, 1.0, 77)
    got = run_gpu(s, 1.0, 77)
    assert_parity(s, 1.0, 77, got, ref)
    for b in range(0, 24, 3):
        assert int(got[0][b]) <= b % 5


def test_sampled_cold_equals_greedy():
    """At a cold temperature on sharp rows the draw is the argmax: the
    sampled kernel must return what greedy verification returns."""
    B, Kp = 40, 5
    t, d, tokens, u = pins._sharp_case(B, Kp, V=64)
    V = t.shape[1]
    s = wl.SampledInputs(B=B, Kp=Kp, V=V, target_logits=t, draft_logits=d, tokens=tokens,
                         u_accept=u)
    acc, bon = run_gpu(s, 0.01, 11)
    gacc = torch.empty(B, dtype=torch.int32, device="cuda")
    gbon = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = _native.new_workspace(B * (Kp + 1), B)
    _native.verify_greedy(t.cuda(), Kp, tokens.cuda(), gacc, gbon, ws,
                          _native.new_error_word())
    assert torch.equal(acc, gacc.cpu()) and torch.equal(bon, gbon.cpu())
    racc, rbon = run_oracle(s, 0.01, 11)
    assert torch.equal(acc, racc) and torch.equal(bon, rbon)


def test_sampled_same_distribution_accepts_all():
    s = wl.make_sampled_inputs(48, 6, 4099, dtype=torch.bfloat16, seed=12)
    s.draft_logits.view(48, 6, 4099).copy_(s.target_logits.view(48, 7, 4099)[:, :6])
    acc, bon = run_gpu(s, 0.7, 5)
    assert (acc == 6).all()
    assert_parity(s, 0.7, 5, (acc, bon), run_oracle(s, 0.7, 5))


def _chi2(counts, probs):
    n = counts.sum()
    exp = probs * n
    return float(((counts - exp) ** 2 / exp).sum())


def test_sampled_preserves_target_distribution():
    """First emitted token ~ p_0 whatever the drafter proposes; after an
    accepted draft the bonus ~ p_1; a plain draw ~ p_0 (chi-square, 3
    degrees of freedom, 99.9 % quantile 16.27, 40000 requests)."""
    rng = np.random.default_rng(23)
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
    s = wl.SampledInputs(B=N, Kp=1, V=V, target_logits=t, draft_logits=d, tokens=tokens,
                         u_accept=u)
    acc, bon = run_gpu(s, 1.0, 4242)
    acc, bon = acc.numpy(), bon.numpy()
    first = np.where(acc >= 1, x, bon)
    assert _chi2(np.bincount(first, minlength=V), p0) < 16.27
    assert _chi2(np.bincount(bon[acc == 1], minlength=V), p1) < 16.27
    s0 = wl.SampledInputs(B=N, Kp=0, V=V, target_logits=t[0::2].contiguous(),
                          draft_logits=torch.empty(0, V), tokens=torch.empty(0, dtype=torch.int32),
                          u_accept=torch.empty(0))
    _, bon0 = run_gpu(s0, 1.0, 99)
    assert _chi2(np.bincount(bon0.numpy(), minlength=V), p0) < 16.27


def test_sampled_residual_across_chunks():
    """A wide row whose support is four far-apart columns (the residual
    weight 0.2 and 0.3 sits in columns 1 and 2049, in different residual
    units): the first emitted token must still follow p_0 over them, and
    every request equals the oracle up to explained near ties."""
    rng = np.random.default_rng(31)
    N, V = 4000, 4096
    cols = np.array([0, 2048, 1, 2049])
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
    s = wl.SampledInputs(B=N, Kp=1, V=V, target_logits=t, draft_logits=d, tokens=tokens,
                         u_accept=u)
    got = run_gpu(s, 1.0, 4343)
    assert_parity(s, 1.0, 4343, got, run_oracle(s, 1.0, 4343))
    acc, bon = got[0].numpy(), got[1].numpy()
    first = np.where(acc >= 1, x, bon)
    assert np.isin(first, cols).all()
    counts = np.array([(first == c).sum() for c in cols])
    assert _chi2(counts, p0) < 16.27


def test_sampled_workspace_reuse_and_determinism():
    big = wl.make_sampled_inputs(64, 7, 20011, dtype=torch.bfloat16, seed=13)
    small = wl.make_sampled_inputs(5, 2, 999, dtype=torch.float32, seed=14)
    ws = torch.zeros(_native.workspace_bytes_sampled(64, 7), dtype=torch.uint8, device="cuda")
    first = run_gpu(big, 1.0, 31, workspace=ws)
    mid = run_gpu(small, 1.0, 32, workspace=ws)
    again = run_gpu(big, 1.0, 31, workspace=ws)
    assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    assert_parity(small, 1.0, 32, mid, run_oracle(small, 1.0, 32))
    other = run_gpu(big, 1.0, 32, workspace=ws)  # another seed draws other tokens
    assert torch.equal(first[0], other[0])       # the accept coins are the caller's
    assert not torch.equal(first[1], other[1])


def test_sampled_argument_errors():
    s = wl.make_sampled_inputs(2, 1, 64, dtype=torch.float32, seed=15).to("cuda")
    acc = torch.empty(2, dtype=torch.int32, device="cuda")
    bon = torch.empty(2, dtype=torch.int32, device="cuda")
    ws = torch.zeros(_native.workspace_bytes_sampled(2, 1), dtype=torch.uint8, device="cuda")
    err = _native.new_error_word()
    for T in (0.0, -1.0, float("nan")):
        with pytest.raises(_native.PEError):
            _native.verify_sampled(s.target_logits, s.draft_logits, 1, s.tokens, s.u_accept,
                                   T, 1, acc, bon, ws, err)
    with pytest.raises(_native.PEError):  # misaligned row stride (63 floats)
        tl = torch.zeros(4, 63, device="cuda")
        _native.verify_sampled(tl, s.draft_logits[:, :63], 1, s.tokens, s.u_accept, 1.0, 1,
                               acc, bon, ws, err)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0


# Seeded random shapes: batch, draft depth (0 included), vocabulary (ragged
# tails, below one vector, many chunks), element type and temperature all
# drawn from one generator per case.
@pytest.mark.parametrize("case", range(24))
def test_sampled_fuzz(case):
    rng = np.random.default_rng(4242 + case)
    B = int(rng.integers(1, 33))
    Kp = int(rng.integers(0, 9))
    V = int(rng.choice([int(rng.integers(1, 9)), int(rng.integers(9, 3000)),
                        int(rng.integers(3000, 70001))]))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    T = float(rng.choice([0.3, 0.7, 1.0, 1.6, 3.0]))
    s = wl.make_sampled_inputs(B, Kp, V, dtype=dtype, seed=3000 + case)
    seed = int(rng.integers(0, 2**63))
    ref = run_oracle(s, T, seed)
    got = run_gpu(s, T, seed)
    assert_parity(s, T, seed, got, ref)
