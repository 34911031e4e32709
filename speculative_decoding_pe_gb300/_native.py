"""ctypes binding of libpe.so (argument marshalling only).

Every function takes torch CUDA tensors, checks their dtype / device /
layout, and passes raw pointers plus the current CUDA stream to the C ABI
declared in ``include/pe_api.h``.  All work runs in the library's kernels;
there is no fallback of any kind: if the library is missing or a call is
rejected, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpe.so")
# the same ABI compiled with PE_CHECKED (NaN logits and internal invariants
# raise ERR_NAN / ERR_INTERNAL; slower, for debugging)
CHECKED_LIB_PATH = os.path.join(_HERE, "_build", "libpe_checked.so")

PE_F32, PE_BF16 = 0, 1
ERR_TOKEN_RANGE = 1
ERR_BLOCK_RANGE = 2
ERR_SLOT_RANGE = 4
ERR_OFFSETS = 8
ERR_MAP_RANGE = 16
ERR_TIMEOUT = 32
ERR_ROW_RANGE = 64
ERR_NAN = 128
ERR_INTERNAL = 256
ERR_WORKSPACE = 512
MAX_KP, MAX_K = 255, 256

# every function the C header declares
EXPORTS = ("pe_workspace_bytes", "pe_verify_greedy", "pe_draft_readout",
           "pe_workspace_bytes_sampled", "pe_verify_sampled",
           "pe_build_draft_batch",
           "pe_assemble_draft_inputs", "pe_step", "pe_step_early_exit", "pe_step_noalloc",
           "pe_get_tuning",
           "pe_set_tuning", "pe_latency_floor", "pe_status_str")


class PEError(RuntimeError):
    def __init__(self, status: int, what: str, lib=None):
        name = lib.pe_status_str(status).decode() if lib is not None else str(status)
        super().__init__("%s failed: %s" % (what, name))
        self.status = status


P = ctypes.c_void_p
i32, i64 = ctypes.c_int32, ctypes.c_int64


class StepArgs(ctypes.Structure):
    """Mirror of pe_step_args."""
    _fields_ = [("B", i32), ("Kp", i32), ("K", i32), ("V", i32), ("H", i32), ("R", i32),
                ("mask_id", i32), ("bt_width", i32), ("block_size", i32),
                ("logits_dtype", i32), ("x_dtype", i32),
                ("logits_row_stride", i64),
                ("logits", P), ("in_offsets", P), ("in_tokens", P), ("in_positions", P),
                ("block_table", P), ("emb", P), ("target_hidden", P), ("h_shared", P),
                ("accepted_len", P), ("bonus_token", P), ("target_argmax", P),
                ("out_offsets", P), ("out_tokens", P), ("out_positions", P),
                ("is_rejected", P), ("is_masked", P), ("hidden_map", P),
                ("slot_mapping", P), ("sample_idx", P), ("X", P),
                ("workspace", P), ("err", P)]


class Tuning(ctypes.Structure):
    """Mirror of pe_tuning."""
    _fields_ = [("ctas_per_sm", i32), ("chunk_batches", i32), ("rows_per_unit", i32),
                ("variant", i32), ("queue_order", i32), ("early_full_read_mb", i32),
                ("single_pass", i32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load():
    """Load libpe.so; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIB_PATH)
        return _lib


_checked = None


def load_checked():
    """Load libpe_checked.so (same entry points, PE_CHECKED); raise if absent."""
    global _checked
    with _lock:
        if _checked is None:
            _checked = _open(CHECKED_LIB_PATH)
        return _checked


def _open(path: str):
    if not os.path.exists(path):
        raise RuntimeError(
            "%s is not built; run speculative_decoding_pe_gb300.build.build() first -- "
            "there is no fallback path" % path)
    lib = ctypes.CDLL(path)
    lib.pe_workspace_bytes.argtypes = [i32, i32]
    lib.pe_workspace_bytes.restype = ctypes.c_size_t
    lib.pe_verify_greedy.argtypes = [P, ctypes.c_int, i64, i32, i32, i32, P, P, P,
                                     P, P, P, P]
    lib.pe_draft_readout.argtypes = [P, ctypes.c_int, i64, i32, i32, P, i32, P, P, P, P]
    lib.pe_draft_readout.restype = ctypes.c_int
    lib.pe_workspace_bytes_sampled.argtypes = [i32, i32]
    lib.pe_workspace_bytes_sampled.restype = ctypes.c_size_t
    lib.pe_verify_sampled.argtypes = [P, P, ctypes.c_int, i64, i64, i32, i32, i32, P, P,
                                      ctypes.c_float, ctypes.c_uint64, P, P, P, P, P]
    lib.pe_verify_sampled.restype = ctypes.c_int
    lib.pe_build_draft_batch.argtypes = ([i32, i32, i32, i32, i32, P, P, P, P, P, P,
                                          i32, i32] + [P] * 10)
    lib.pe_assemble_draft_inputs.argtypes = [ctypes.c_int, i32, i32, i32, i32] + [P] * 9
    lib.pe_step.argtypes = [ctypes.POINTER(StepArgs), P]
    lib.pe_step_early_exit.argtypes = [ctypes.POINTER(StepArgs), P]
    lib.pe_step_early_exit.restype = ctypes.c_int
    lib.pe_step_noalloc.argtypes = [ctypes.POINTER(StepArgs), P]
    lib.pe_step_noalloc.restype = ctypes.c_int
    lib.pe_get_tuning.argtypes = [ctypes.POINTER(Tuning)]
    lib.pe_set_tuning.argtypes = [ctypes.POINTER(Tuning)]
    lib.pe_latency_floor.argtypes = [i32, i32, P, i32, P, P]
    lib.pe_latency_floor.restype = ctypes.c_int
    lib.pe_status_str.argtypes = [ctypes.c_int]
    lib.pe_status_str.restype = ctypes.c_char_p
    for f in ("pe_verify_greedy", "pe_build_draft_batch", "pe_assemble_draft_inputs",
              "pe_step", "pe_get_tuning", "pe_set_tuning"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


# ------------------------------------------------------------------ helpers

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PE_F32
    if t.dtype == torch.bfloat16:
        return PE_BF16
    raise TypeError("expected float32 or bfloat16, got %s" % t.dtype)


def _dev(t: torch.Tensor | None, name: str, dtype=None, numel=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if numel is not None and t.numel() < numel:
        raise ValueError("%s holds %d elements, needs %d" % (name, t.numel(), numel))
    return ctypes.c_void_p(t.data_ptr())


def _logits(t: torch.Tensor):
    if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("logits must be a 2-D CUDA tensor with unit column stride")
    return ctypes.c_void_p(t.data_ptr()), _dtype_code(t), t.stride(0)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(lib, rc: int, what: str):
    if rc != 0:
        raise PEError(rc, what, lib)


# ---------------------------------------------------------------- public API

def workspace_bytes(logits_rows: int, B: int) -> int:
    return int(load().pe_workspace_bytes(logits_rows, B))


def new_workspace(logits_rows: int, B: int, device="cuda") -> torch.Tensor:
    """Zero-filled scratch for verify_greedy / step (reusable across calls)."""
    return torch.zeros(workspace_bytes(logits_rows, B), dtype=torch.uint8, device=device)


def new_error_word(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def verify_greedy(logits, Kp, in_tokens, accepted_len, bonus_token, workspace, err,
                  target_argmax=None, stream=None):
    """Greedy verification of B requests (rows B*(Kp+1) of ``logits``)."""
    lib = load()
    lp, dt, stride = _logits(logits)
    rows = logits.shape[0]
    if rows % (Kp + 1):
        raise ValueError("logits rows must be a multiple of Kp+1")
    B = rows // (Kp + 1)
    rc = lib.pe_verify_greedy(
        lp, dt, stride, B, Kp, logits.shape[1],
        _dev(in_tokens, "in_tokens", torch.int32, rows if Kp else None),
        _dev(accepted_len, "accepted_len", torch.int32, B),
        _dev(bonus_token, "bonus_token", torch.int32, B),
        _dev(target_argmax, "target_argmax", torch.int32, rows),
        _dev(workspace, "workspace", torch.uint8, workspace_bytes(rows, B)),
        _dev(err, "err", torch.int32, 1), _stream(stream))
    _check(lib, rc, "pe_verify_greedy")


def workspace_bytes_sampled(B: int, Kp: int) -> int:
    return int(load().pe_workspace_bytes_sampled(B, Kp))


def verify_sampled(target_logits, draft_logits, Kp, in_tokens, u_accept, temperature, seed,
                   accepted_len, bonus_token, workspace, err, stream=None):
    """Rejection-sampling verification of B requests: target rows B*(Kp+1),
    draft rows B*Kp, accept coins u_accept[B*Kp], Philox seed for the draws."""
    lib = load()
    tp, dt, tstride = _logits(target_logits)
    rows, V = target_logits.shape
    if rows % (Kp + 1):
        raise ValueError("target_logits rows must be a multiple of Kp+1")
    B = rows // (Kp + 1)
    if Kp:
        dp, ddt, dstride = _logits(draft_logits)
        if ddt != dt or draft_logits.shape[1] != V or draft_logits.shape[0] < B * Kp:
            raise ValueError("draft_logits must be [B*Kp, V] of the target's dtype")
    else:
        dp, dstride = None, 0
    rc = lib.pe_verify_sampled(
        tp, dp, dt, tstride, dstride, B, Kp, V,
        _dev(in_tokens, "in_tokens", torch.int32, rows if Kp else None),
        _dev(u_accept, "u_accept", torch.float32, B * Kp if Kp else None),
        float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF,
        _dev(accepted_len, "accepted_len", torch.int32, B),
        _dev(bonus_token, "bonus_token", torch.int32, B),
        _dev(workspace, "workspace", torch.uint8, workspace_bytes_sampled(B, Kp)),
        _dev(err, "err", torch.int32, 1), _stream(stream))
    _check(lib, rc, "pe_verify_sampled")


def draft_readout(logits, out_tokens, workspace, err, sample_idx=None, stream=None):
    """Greedy draft tokens: argmax of logits row sample_idx[i] (row i when
    sample_idx is None) into out_tokens[i]."""
    lib = load()
    lp, dt, stride = _logits(logits)
    rows, V = logits.shape
    n = sample_idx.numel() if sample_idx is not None else out_tokens.numel()
    rc = lib.pe_draft_readout(
        lp, dt, stride, rows, V, _dev(sample_idx, "sample_idx", torch.int32, n), n,
        _dev(out_tokens, "out_tokens", torch.int32, n),
        _dev(workspace, "workspace", torch.uint8, workspace_bytes(n, n)),
        _dev(err, "err", torch.int32, 1), _stream(stream))
    _check(lib, rc, "pe_draft_readout")


@dataclass
class DraftBatch:
    """Outputs of the rebuild (and of the fused step)."""
    out_offsets: torch.Tensor
    out_tokens: torch.Tensor
    out_positions: torch.Tensor
    is_rejected: torch.Tensor
    is_masked: torch.Tensor
    hidden_map: torch.Tensor
    slot_mapping: torch.Tensor
    sample_idx: torch.Tensor | None

    @staticmethod
    def empty(B, K, R, device="cuda", sample_idx=True):
        T = R + B * (K - 1)
        e = lambda n, dt: torch.empty(n, dtype=dt, device=device)
        return DraftBatch(e(B + 1, torch.int32), e(T, torch.int32), e(T, torch.int32),
                          e(T, torch.uint8), e(T, torch.uint8), e(R, torch.int32),
                          e(T, torch.int64), e(B * K, torch.int32) if sample_idx else None)


def build_draft_batch(B, Kp, K, mask_id, R, in_offsets, in_tokens, in_positions,
                      accepted_len, bonus_token, block_table, block_size, out: DraftBatch,
                      err, stream=None):
    lib = load()
    T = R + B * (K - 1)
    if block_table.dim() != 2 or block_table.shape[0] < B:
        raise ValueError("block_table must be [B, width]")
    rc = lib.pe_build_draft_batch(
        B, Kp, K, mask_id, R, _dev(in_offsets, "in_offsets", torch.int32, B + 1),
        _dev(in_tokens, "in_tokens", torch.int32, R),
        _dev(in_positions, "in_positions", torch.int32, R),
        _dev(accepted_len, "accepted_len", torch.int32, B),
        _dev(bonus_token, "bonus_token", torch.int32, B),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1], block_size,
        _dev(out.out_offsets, "out_offsets", torch.int32, B + 1),
        _dev(out.out_tokens, "out_tokens", torch.int32, T),
        _dev(out.out_positions, "out_positions", torch.int32, T),
        _dev(out.is_rejected, "is_rejected", torch.uint8, T),
        _dev(out.is_masked, "is_masked", torch.uint8, T),
        _dev(out.hidden_map, "hidden_map", torch.int32, R),
        _dev(out.slot_mapping, "slot_mapping", torch.int64, T),
        _dev(out.sample_idx, "sample_idx", torch.int32, B * K),
        _dev(err, "err", torch.int32, 1), _stream(stream))
    _check(lib, rc, "pe_build_draft_batch")


def assemble_draft_inputs(emb, target_hidden, h_shared, out_tokens, hidden_map,
                          is_masked, X, err, stream=None):
    lib = load()
    V, H = emb.shape
    T, R = out_tokens.numel(), hidden_map.numel()
    dt = _dtype_code(emb)
    for name, t in (("target_hidden", target_hidden), ("h_shared", h_shared), ("X", X)):
        if t.dtype != emb.dtype:
            raise TypeError("%s must match the embedding dtype" % name)
    rc = lib.pe_assemble_draft_inputs(
        dt, H, V, T, R, _dev(emb, "emb"), _dev(target_hidden, "target_hidden", None, R * H),
        _dev(h_shared, "h_shared", None, H), _dev(out_tokens, "out_tokens", torch.int32),
        _dev(hidden_map, "hidden_map", torch.int32), _dev(is_masked, "is_masked", torch.uint8, T),
        _dev(X, "X", None, T * 2 * H), _dev(err, "err", torch.int32, 1), _stream(stream))
    _check(lib, rc, "pe_assemble_draft_inputs")


@dataclass
class StepOutputs(DraftBatch):
    accepted_len: torch.Tensor = None
    bonus_token: torch.Tensor = None
    target_argmax: torch.Tensor | None = None
    X: torch.Tensor = None

    @staticmethod
    def empty(B, Kp, K, R, H, dtype, device="cuda", sample_idx=True, target_argmax=True):
        d = DraftBatch.empty(B, K, R, device, sample_idx)
        T = R + B * (K - 1)
        return StepOutputs(**d.__dict__,
                           accepted_len=torch.empty(B, dtype=torch.int32, device=device),
                           bonus_token=torch.empty(B, dtype=torch.int32, device=device),
                           target_argmax=(torch.empty(B * (Kp + 1), dtype=torch.int32,
                                                      device=device) if target_argmax else None),
                           X=torch.empty(T, 2 * H, dtype=dtype, device=device))


def make_step_args(*, logits, Kp, K, mask_id, in_offsets, in_tokens, in_positions,
                   block_table, block_size, emb, target_hidden, h_shared,
                   out: StepOutputs, workspace, err) -> StepArgs:
    """Check the tensors once and pack a pe_step_args (reusable while the
    same tensors stay alive)."""
    lp, ldt, stride = _logits(logits)
    V, H = emb.shape
    if logits.shape[1] != V:
        raise ValueError("logits width must equal the vocabulary size")
    rows = logits.shape[0]
    if rows % (Kp + 1):
        raise ValueError("logits rows must be a multiple of Kp+1")
    B = rows // (Kp + 1)
    R = in_tokens.numel()
    T = R + B * (K - 1)
    a = StepArgs()
    a.B, a.Kp, a.K, a.V, a.H, a.R = B, Kp, K, V, H, R
    a.mask_id, a.bt_width, a.block_size = mask_id, block_table.shape[1], block_size
    a.logits_dtype, a.x_dtype = ldt, _dtype_code(emb)
    a.logits_row_stride = stride
    a.logits = lp
    a.in_offsets = _dev(in_offsets, "in_offsets", torch.int32, B + 1)
    a.in_tokens = _dev(in_tokens, "in_tokens", torch.int32, R)
    a.in_positions = _dev(in_positions, "in_positions", torch.int32, R)
    a.block_table = _dev(block_table, "block_table", torch.int32)
    a.emb = _dev(emb, "emb")
    a.target_hidden = _dev(target_hidden, "target_hidden", emb.dtype, R * H)
    a.h_shared = _dev(h_shared, "h_shared", emb.dtype, H)
    a.accepted_len = _dev(out.accepted_len, "accepted_len", torch.int32, B)
    a.bonus_token = _dev(out.bonus_token, "bonus_token", torch.int32, B)
    a.target_argmax = _dev(out.target_argmax, "target_argmax", torch.int32, rows)
    a.out_offsets = _dev(out.out_offsets, "out_offsets", torch.int32, B + 1)
    a.out_tokens = _dev(out.out_tokens, "out_tokens", torch.int32, T)
    a.out_positions = _dev(out.out_positions, "out_positions", torch.int32, T)
    a.is_rejected = _dev(out.is_rejected, "is_rejected", torch.uint8, T)
    a.is_masked = _dev(out.is_masked, "is_masked", torch.uint8, T)
    a.hidden_map = _dev(out.hidden_map, "hidden_map", torch.int32, R)
    a.slot_mapping = _dev(out.slot_mapping, "slot_mapping", torch.int64, T)
    a.sample_idx = _dev(out.sample_idx, "sample_idx", torch.int32, B * K)
    a.X = _dev(out.X, "X", emb.dtype, T * 2 * H)
    a.workspace = _dev(workspace, "workspace", torch.uint8, workspace_bytes(rows, B))
    a.err = _dev(err, "err", torch.int32, 1)
    return a


def step_packed(args: StepArgs, stream=None):
    """Launch the fused step from a packed argument block."""
    lib = load()
    _check(lib, lib.pe_step(ctypes.byref(args), _stream(stream)), "pe_step")


def step_early_exit_packed(args: StepArgs, stream=None):
    """The fused step with early exit (rows after each request's first
    mismatch are not read; target_argmax holds -1 for them)."""
    lib = load()
    _check(lib, lib.pe_step_early_exit(ctypes.byref(args), _stream(stream)),
           "pe_step_early_exit")


def step(**kw):
    """The whole step (verify, rebuild, assemble) in one launch; see
    make_step_args for the arguments and an optional ``stream``."""
    stream = kw.pop("stream", None)
    step_packed(make_step_args(**kw), stream)


def latency_floor(ctas: int, hops: int = 0, chain=None, out=None, stream=None):
    """An empty launch of ``ctas`` CTAs, plus ``hops`` dependent loads through
    ``chain`` (int32, entry i = index of the next) ending in ``out[0]``."""
    lib = load()
    n = chain.numel() if chain is not None else 0
    rc = lib.pe_latency_floor(ctas, hops, _dev(chain, "chain", torch.int32), n,
                              _dev(out, "out", torch.int32, 1), _stream(stream))
    _check(lib, rc, "pe_latency_floor")


def get_tuning() -> dict:
    lib = load()
    t = Tuning()
    _check(lib, lib.pe_get_tuning(ctypes.byref(t)), "pe_get_tuning")
    return {f: getattr(t, f) for f, _ in Tuning._fields_}


def set_tuning(**kw):
    lib = load()
    t = Tuning(**{f: int(kw.get(f, 0)) for f, _ in Tuning._fields_})
    _check(lib, lib.pe_set_tuning(ctypes.byref(t)), "pe_set_tuning")
