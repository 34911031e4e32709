"""Seeded synthetic workloads for the P-EAGLE drafting step.

This module draws random inputs and nothing else: it holds none of the step's
arithmetic (no argmax, no acceptance rule, no rebuild, no gather).  Both the
CUDA path and the CPU oracle consume what it produces.

Acceptance lengths are *planted*: every random logit is clamped to
[-CLAMP, CLAMP] and, for request b with planted length a_b, row j < a_b gets
PLANT at the column of draft d_{j+1}; row a_b (when a_b < K') gets PLANT at a
column chosen different from d_{a_b+1}.  PLANT > CLAMP, so the planted column
is the unique maximum of its row and the planted length is the length any
correct greedy verifier must find.  Rows after a_b stay purely random (their
argmax, including ties, is left to the implementation under test).

Workload shapes follow the pages' workloads (GPT-OSS-20B-shaped and
Qwen3-Coder-30B-shaped decode, first draft after prefill); the pages'
benchmark suites (MT-Bench, HumanEval, SPEED-Bench) are stood in for by
geometric accept-length distributions with means near the pages' acceptance
lengths.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch

PLANT = 64.0    # exactly representable in bf16 and fp32
CLAMP = 32.0    # |random logit| <= CLAMP < PLANT


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    description: str
    B: int                  # requests
    Kp: int                 # previous draft depth K' (0: first step after prefill)
    K: int                  # new draft depth
    H: int                  # hidden size
    V: int                  # vocabulary size
    dtype: torch.dtype      # logits, embedding table, hidden states, X
    emb_std: float
    hidden_std: float
    logits_std: float
    accept_p: float = 0.0   # geometric(p): failures before first success
    zero_frac: float = 0.0  # fraction of requests forced to accept nothing
    forced: tuple = ()      # ((request, accepted_len), ...)
    start_lo: int = 0       # first position of a decode segment, U[lo, hi)
    start_hi: int = 1
    prompt_lo: int = 0      # prefill prompt length, U[lo, hi] inclusive
    prompt_hi: int = 0
    bt_width: int = 1       # block-table columns per request
    bt_per_row: bool = False  # each row its own permutation of bt_width ids
    block_size: int = 16
    row_pad: int = 0        # extra logits columns per row (misaligned V tests)

    @property
    def mask_id(self) -> int:
        return self.V - 1

    @property
    def prefill(self) -> bool:
        return self.Kp == 0

    def with_(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


def _w(max_pos: int, bs: int = 16) -> int:
    return max_pos // bs + 1


SPECS = {
    "tiny": WorkloadSpec(
        "tiny", "tiny fp32 case: B=4 K'=3 K=3 H=64 V=1000",
        B=4, Kp=3, K=3, H=64, V=1000, dtype=torch.float32,
        emb_std=1.0, hidden_std=1.0, logits_std=1.0, accept_p=0.35,
        start_lo=0, start_hi=512, bt_width=64, bt_per_row=True),
    "decode_b1": WorkloadSpec(
        "decode_b1", "single-stream decode B=1 K'=7 K=7 H=2880 V=201088 bf16",
        B=1, Kp=7, K=7, H=2880, V=201088, dtype=torch.bfloat16,
        emb_std=0.02, hidden_std=1.0, logits_std=2.0, accept_p=0.25,
        start_lo=1024, start_hi=8192, bt_width=_w(8191 + 7 + 6)),
    "decode_b64": WorkloadSpec(
        "decode_b64", "decode B=64 K'=7 K=7 H=2880 V=201088 bf16",
        B=64, Kp=7, K=7, H=2880, V=201088, dtype=torch.bfloat16,
        emb_std=0.02, hidden_std=1.0, logits_std=2.0, accept_p=0.3,
        forced=((0, 7), (1, 0)), start_lo=256, start_hi=32768,
        bt_width=_w(32767 + 7 + 6)),
    "prefill_b8": WorkloadSpec(
        "prefill_b8", "first draft after prefill B=8 L~U[1024,8192] K=7 H=2880 "
        "V=201088 bf16", B=8, Kp=0, K=7, H=2880, V=201088, dtype=torch.bfloat16,
        emb_std=0.02, hidden_std=1.0, logits_std=2.0, prompt_lo=1024,
        prompt_hi=8192, bt_width=_w(8191 + 6)),
    "decode_b256": WorkloadSpec(
        "decode_b256", "large-batch decode B=256 K'=7 K=7 H=2048 V=151936 bf16",
        B=256, Kp=7, K=7, H=2048, V=151936, dtype=torch.bfloat16,
        emb_std=0.02, hidden_std=1.0, logits_std=2.0, accept_p=0.2,
        zero_frac=0.4, start_lo=0, start_hi=65536, bt_width=_w(65535 + 7 + 6)),
}


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    logits: torch.Tensor          # [B*(Kp+1), V] view (row stride may exceed V)
    in_offsets: torch.Tensor | None  # [B+1] int32 (prefill only)
    in_tokens: torch.Tensor       # [R] int32
    in_positions: torch.Tensor    # [R] int32
    block_table: torch.Tensor     # [B, W] int32
    emb: torch.Tensor             # [V, H]
    hidden: torch.Tensor          # [R, H]
    h_shared: torch.Tensor        # [H]
    planted_accept: torch.Tensor  # [B] int32 (prefill: zeros)
    planted_bonus: torch.Tensor   # [B] int32, -1 where not planted
    extra: dict = field(default_factory=dict)

    # sizes in the step's notation
    @property
    def B(self): return self.spec.B
    @property
    def Kp(self): return self.spec.Kp
    @property
    def K(self): return self.spec.K
    @property
    def V(self): return self.spec.V
    @property
    def H(self): return self.spec.H
    @property
    def mask_id(self): return self.spec.mask_id
    @property
    def block_size(self): return self.spec.block_size
    @property
    def R(self): return self.in_tokens.numel()
    @property
    def T(self): return self.R + self.B * (self.K - 1)
    @property
    def logits_rows(self): return self.B * (self.Kp + 1)

    def to(self, device) -> "Workload":
        """Copy every tensor to ``device`` (the logits keep their row stride)."""
        kw = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = _move(v, device)
        kw["extra"] = dict(self.extra)
        return Workload(**kw)


def _move(t: torch.Tensor, device) -> torch.Tensor:
    """Copy to ``device``; a 2-D view with padded rows keeps its row stride
    and the padding's contents."""
    if t.dim() == 2 and t.stride(1) == 1 and t.shape[0] and t.stride(0) != t.shape[1]:
        base = torch.empty(t.shape[0], t.stride(0), dtype=t.dtype, device=device)
        base.copy_(t.as_strided((t.shape[0], t.stride(0)), (t.stride(0), 1)))
        return base[:, : t.shape[1]]
    return t.to(device).contiguous()


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _randint(lo, hi, shape, g, device):
    return torch.randint(lo, hi, shape, generator=g, device=device, dtype=torch.int64)


def _geometric(p: float, g) -> int:
    """Failures before the first success of Bernoulli(p) trials."""
    u = torch.rand((), generator=g).item()
    return int(math.floor(math.log1p(-u) / math.log1p(-p))) if p < 1.0 else 0


def make_workload(spec: WorkloadSpec | str, seed: int = 0, device="cpu") -> Workload:
    """Draw one seeded workload on ``device``.

    Shared tensors (embedding table, h_shared, block table, prompt lengths)
    come from one generator; each request's rows (tokens, start position,
    accept length, logits, hidden states) from a generator of its own, so a
    request can be re-drawn alone."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    device = torch.device(device)
    B, Kp, K, H, V = spec.B, spec.Kp, spec.K, spec.H, spec.V
    dt = spec.dtype
    base_seed = int(seed) * 1_000_003
    gs_cpu = _gen("cpu", base_seed)           # scalars drawn on the host
    gs = _gen(device, base_seed + 7)          # shared tensors

    emb = _randn((V, H), spec.emb_std, gs, device).to(dt)
    h_shared = _randn((H,), 1.0, gs, device).to(dt)

    if spec.prefill:
        lens = [int(_randint(spec.prompt_lo, spec.prompt_hi + 1, (), gs_cpu, "cpu"))
                for _ in range(B)]
    else:
        lens = [Kp + 1] * B
    R = sum(lens)
    W = spec.bt_width
    if spec.bt_per_row:
        bt = torch.stack([torch.randperm(W, generator=gs, device=device)
                          for _ in range(B)]) if B else torch.empty(0, W, device=device)
    else:
        bt = torch.randperm(B * W, generator=gs, device=device).view(B, W)
    bt = bt.to(torch.int32)

    n_lrows = B * (Kp + 1)
    stride = V + spec.row_pad
    logits_base = torch.empty((n_lrows, stride), dtype=dt, device=device)
    if spec.row_pad:
        logits_base[:, V:] = 2 * PLANT   # any read past V would win the argmax
    tokens = torch.empty(R, dtype=torch.int32, device=device)
    positions = torch.empty(R, dtype=torch.int32, device=device)
    hidden = torch.empty((R, H), dtype=dt, device=device)
    planted_a = torch.zeros(B, dtype=torch.int32)
    planted_bonus = torch.full((B,), -1, dtype=torch.int32)
    forced = dict(spec.forced)

    row = 0
    for b in range(B):
        n = lens[b]
        g_cpu = _gen("cpu", base_seed + 1000 + 2 * b)
        g = _gen(device, base_seed + 1001 + 2 * b)
        toks = _randint(0, V - 1, (n,), g, device)  # MASK id V-1 never drawn
        hidden[row:row + n] = _randn((n, H), spec.hidden_std, g, device).to(dt)
        lg = _randn((Kp + 1, V), spec.logits_std, g, device).clamp_(-CLAMP, CLAMP)
        if spec.prefill:
            start = 0
        else:
            start = int(_randint(spec.start_lo, spec.start_hi, (), g_cpu, "cpu"))
            if b in forced:
                a = forced[b]
            elif spec.zero_frac and torch.rand((), generator=g_cpu).item() < spec.zero_frac:
                a = 0
            else:
                a = min(_geometric(spec.accept_p, g_cpu), Kp)
            planted_a[b] = a
            d = toks[1:].tolist()            # drafts d_1..d_K'
            cols = list(d[:a])
            if a < Kp:
                t = int(_randint(0, V - 1, (), g_cpu, "cpu"))
                if t >= d[a]:
                    t += 1                   # uniform over columns != d_{a+1}
                cols.append(t)
                planted_bonus[b] = t
            for j, c in enumerate(cols):
                lg[j, c] = PLANT
        tokens[row:row + n] = toks.to(torch.int32)
        positions[row:row + n] = torch.arange(start, start + n, device=device,
                                              dtype=torch.int32)
        logits_base[b * (Kp + 1):(b + 1) * (Kp + 1), :V] = lg.to(dt)
        row += n

    in_offsets = None
    if spec.prefill:
        in_offsets = torch.tensor([0] + lens, dtype=torch.int64).cumsum(0).to(
            device=device, dtype=torch.int32)
    return Workload(spec=spec, seed=seed, logits=logits_base[:, :V],
                    in_offsets=in_offsets, in_tokens=tokens, in_positions=positions,
                    block_table=bt, emb=emb, hidden=hidden, h_shared=h_shared,
                    planted_accept=planted_a, planted_bonus=planted_bonus,
                    extra={"prompt_lens": lens})


@dataclass
class SampledInputs:
    """Inputs of rejection-sampling verification (request-major rows)."""
    B: int
    Kp: int
    V: int
    target_logits: torch.Tensor   # [B*(Kp+1), V]
    draft_logits: torch.Tensor    # [B*Kp, V] (a [0, V] tensor when Kp == 0)
    tokens: torch.Tensor          # [B*(Kp+1)] int32; row j+1 holds draft d_{j+1}
    u_accept: torch.Tensor        # [B*Kp] float32 in [0, 1)

    def to(self, device) -> "SampledInputs":
        kw = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = _move(v, device)
        return SampledInputs(**kw)


def make_sampled_inputs(B: int, Kp: int, V: int, dtype=torch.bfloat16, seed: int = 0,
                        logits_std: float = 2.0, draft_noise: float = 0.5,
                        plant: float = 6.0, plant_frac: float = 0.7,
                        device="cpu") -> SampledInputs:
    """Seeded inputs for rejection-sampling verification.

    Target logits are N(0, logits_std) clamped to [-CLAMP, CLAMP]; the drafter
    row of position j is the target row j plus N(0, draft_noise) (a drafter
    that mostly agrees with its target).  Draft tokens are uniform over the
    vocabulary; with probability ``plant_frac`` a draft's column is raised by
    ``plant`` in both its target and its draft row, so that it carries most
    of both distributions.  Each request draws from a generator of its own.

    Rows are padded to a multiple of 16 bytes; the padding holds 2*PLANT, a
    value that would dominate any distribution a read past V took part in."""
    device = torch.device(device)
    base_seed = int(seed) * 1_000_033 + 17
    epv = 16 // torch.empty((), dtype=dtype).element_size()
    stride = (V + epv - 1) // epv * epv
    tl = torch.full((B * (Kp + 1), stride), 2 * PLANT, dtype=dtype, device=device)[:, :V]
    dl = torch.full((B * Kp, stride), 2 * PLANT, dtype=dtype, device=device)[:, :V]
    tokens = torch.empty(B * (Kp + 1), dtype=torch.int32, device=device)
    u = torch.empty(B * Kp, dtype=torch.float32, device=device)
    for b in range(B):
        g = _gen(device, base_seed + 2 * b)
        g_cpu = _gen("cpu", base_seed + 2 * b + 1)
        t = _randn((Kp + 1, V), logits_std, g, device).clamp_(-CLAMP, CLAMP)
        d = (t[:Kp] + _randn((Kp, V), draft_noise, g, device)).clamp_(-CLAMP, CLAMP)
        toks = _randint(0, V, (Kp + 1,), g, device)
        for j in range(Kp):
            if torch.rand((), generator=g_cpu).item() < plant_frac:
                x = int(toks[j + 1])
                t[j, x] += plant
                d[j, x] += plant
        tl[b * (Kp + 1):(b + 1) * (Kp + 1)] = t.to(dtype)
        dl[b * Kp:(b + 1) * Kp] = d.to(dtype)
        tokens[b * (Kp + 1):(b + 1) * (Kp + 1)] = toks.to(torch.int32)
        u[b * Kp:(b + 1) * Kp] = torch.rand((Kp,), generator=g, device=device)
    return SampledInputs(B=B, Kp=Kp, V=V, target_logits=tl, draft_logits=dl,
                         tokens=tokens, u_accept=u)
