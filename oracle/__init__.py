"""CPU oracle for the P-EAGLE parallel-drafting step (verify, rebuild, assemble).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference arm of ``bench.py`` may import this package.  The
product library never calls it and shares no code with it.

The arithmetic lives in ``pe_oracle.c`` (plain single-threaded C).  This module
only compiles it with gcc when needed and marshals torch CPU tensors through
ctypes.  Every function returns fresh CPU tensors.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pe_oracle.c")
_HDR = os.path.join(_HERE, "pe_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F32, BF16 = 0, 1
ERR_TOKEN_RANGE = 1
ERR_BLOCK_RANGE = 2
ERR_SLOT_RANGE = 4
ERR_OFFSETS = 8
ERR_MAP_RANGE = 16
ERR_ROW_RANGE = 64

_lock = threading.Lock()
_libs: dict = {}
_current = None   # path of the library the module-level functions use


def compile_source(src: str, out: str) -> str:
    """gcc -O2 one C file (plain, no vector intrinsics) into a shared library."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Werror",
           "-I", _HERE, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile liboracle.so when missing or older than its sources."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH)
    if not stale:
        t_lib = os.path.getmtime(_LIB_PATH)
        stale = any(os.path.getmtime(p) > t_lib for p in (_SRC, _HDR))
    if stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def use_library(path: str | None) -> None:
    """Point the module-level functions at another build of pe_oracle.c
    (used by the mutation tests); None restores the default build."""
    global _current
    _current = path


def _load():
    with _lock:
        path = _current or build()
        lib = _libs.get(path)
        if lib is None:
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            c_int = ctypes.c_int
            lib.oracle_argmax_rows.argtypes = [P, c_int, i64, i32, i32, P]
            lib.oracle_verify_greedy.argtypes = [P, c_int, i64, i32, i32, i32,
                                                 P, P, P, P]
            lib.oracle_draft_readout.argtypes = [P, c_int, i64, i32, i32, P, i32, P, P]
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_verify_sampled.argtypes = [P, P, c_int, i64, i64, i32, i32, i32, P, P,
                                                  ctypes.c_float, ctypes.c_uint64, P, P]
            lib.oracle_build_draft_batch.argtypes = (
                [i32, i32, i32, i32, P, P, P, P, P, P, i32, i32] + [P] * 9)
            lib.oracle_assemble_draft_inputs.argtypes = (
                [i32, i32, i32, i32, i32] + [P] * 8)
            lib.oracle_step.argtypes = (
                [c_int, c_int, i32, i32, i32, i32, i32, i32, P, i64, P, P, P, P,
                 i32, i32, P, P, P] + [P] * 13)
            for fn in (lib.oracle_argmax_rows, lib.oracle_verify_greedy,
                       lib.oracle_draft_readout, lib.oracle_verify_sampled,
                       lib.oracle_build_draft_batch,
                       lib.oracle_assemble_draft_inputs, lib.oracle_step):
                fn.restype = ctypes.c_int
            _libs[path] = lib
    return lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("oracle handles float32 and bfloat16 only, got %s" % t.dtype)


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu", "oracle takes CPU tensors"
    return ctypes.c_void_p(t.data_ptr())


def _i32(t):
    if t is None:
        return None
    return t.detach().to("cpu", torch.int32).contiguous()


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError("%s rejected its arguments (rc=%d)" % (what, rc))


def argmax_rows(logits: torch.Tensor, V: int | None = None) -> torch.Tensor:
    """argmax over the first V columns of each row; lowest index on ties."""
    lib = _load()
    logits = logits.detach().cpu()
    assert logits.dim() == 2 and logits.stride(1) == 1
    V = logits.shape[1] if V is None else V
    out = torch.empty(logits.shape[0], dtype=torch.int32)
    _check(lib.oracle_argmax_rows(_ptr(logits), _dt(logits), logits.stride(0),
                                  logits.shape[0], V, _ptr(out)), "argmax_rows")
    return out


def draft_readout(logits, sample_idx=None, n=None):
    """Greedy draft tokens: argmax of logits row sample_idx[i] (row i when
    sample_idx is None).  Returns (tokens[n], error word)."""
    lib = _load()
    logits = logits.detach().cpu()
    assert logits.dim() == 2 and logits.stride(1) == 1
    idx = _i32(sample_idx)
    if n is None:
        n = idx.numel() if idx is not None else logits.shape[0]
    out = torch.empty(n, dtype=torch.int32)
    err = ctypes.c_uint32(0)
    _check(lib.oracle_draft_readout(_ptr(logits), _dt(logits), logits.stride(0),
                                    logits.shape[0], logits.shape[1], _ptr(idx), n,
                                    _ptr(out), ctypes.byref(err)), "draft_readout")
    return out, err.value


def philox4x32_10(counter, key):
    """Philox4x32-10 of a 4-word counter under a 2-word key."""
    lib = _load()
    c = (ctypes.c_uint32 * 4)(*counter)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    lib.oracle_philox4x32_10(c, k, o)
    return list(o)


def verify_sampled(target_logits, draft_logits, B, Kp, tokens, u_accept, temperature,
                   seed):
    """Rejection-sampling verification; returns (accepted_len[B], bonus[B])."""
    lib = _load()
    t = target_logits.detach().cpu()
    assert t.dim() == 2 and t.stride(1) == 1
    d = draft_logits.detach().cpu() if draft_logits is not None else None
    if d is not None:
        assert d.dtype == t.dtype and d.stride(1) == 1
    tok = _i32(tokens)
    u = u_accept.detach().to("cpu", torch.float32).contiguous() if u_accept is not None else None
    acc = torch.empty(B, dtype=torch.int32)
    bon = torch.empty(B, dtype=torch.int32)
    _check(lib.oracle_verify_sampled(
        _ptr(t), _ptr(d), _dt(t), t.stride(0), d.stride(0) if d is not None else 0, B, Kp,
        t.shape[1], _ptr(tok), _ptr(u), float(temperature), int(seed), _ptr(acc), _ptr(bon)),
        "verify_sampled")
    return acc, bon


def verify_greedy(logits, B, Kp, V, tokens):
    """Returns (accepted_len[B], bonus_token[B], target_argmax[B*(Kp+1)])."""
    lib = _load()
    logits = logits.detach().cpu()
    assert logits.dim() == 2 and logits.stride(1) == 1
    tokens = _i32(tokens)
    acc = torch.empty(B, dtype=torch.int32)
    bon = torch.empty(B, dtype=torch.int32)
    amax = torch.empty(B * (Kp + 1), dtype=torch.int32)
    _check(lib.oracle_verify_greedy(_ptr(logits), _dt(logits), logits.stride(0),
                                    B, Kp, V, _ptr(tokens), _ptr(acc), _ptr(bon),
                                    _ptr(amax)), "verify_greedy")
    return acc, bon, amax


def _rebuild_outputs(B, K, R, T):
    return {
        "out_offsets": torch.full((B + 1,), -7, dtype=torch.int32),
        "out_tokens": torch.full((T,), -7, dtype=torch.int32),
        "out_positions": torch.full((T,), -7, dtype=torch.int32),
        "is_rejected": torch.full((T,), 7, dtype=torch.uint8),
        "is_masked": torch.full((T,), 7, dtype=torch.uint8),
        "hidden_map": torch.full((R,), -7, dtype=torch.int32),
        "slot_mapping": torch.full((T,), -7, dtype=torch.int64),
        "sample_idx": torch.full((B * K,), -7, dtype=torch.int32),
    }


def build_draft_batch(B, Kp, K, mask_id, in_offsets, in_tokens, in_positions,
                      accepted_len, bonus_token, block_table, block_size):
    """Returns (outputs dict, error word)."""
    lib = _load()
    in_offsets = _i32(in_offsets)
    R = int(in_offsets[B]) if in_offsets is not None else B * (Kp + 1)
    T = R + B * (K - 1)
    o = _rebuild_outputs(B, K, R, T)
    bt = _i32(block_table)
    err = ctypes.c_uint32(0)
    _check(lib.oracle_build_draft_batch(
        B, Kp, K, mask_id, _ptr(in_offsets), _ptr(_i32(in_tokens)),
        _ptr(_i32(in_positions)), _ptr(_i32(accepted_len)),
        _ptr(_i32(bonus_token)), _ptr(bt), bt.shape[1], block_size,
        _ptr(o["out_offsets"]), _ptr(o["out_tokens"]), _ptr(o["out_positions"]),
        _ptr(o["is_rejected"]), _ptr(o["is_masked"]), _ptr(o["hidden_map"]),
        _ptr(o["slot_mapping"]), _ptr(o["sample_idx"]), ctypes.byref(err)),
        "build_draft_batch")
    return o, err.value


def assemble_draft_inputs(H, V, emb, target_hidden, h_shared, out_tokens,
                          hidden_map, is_masked, X=None):
    """X[T, 2H] = emb(tok) (+) hidden; X (if given) supplies the prior content
    of slots that are neither mapped nor masked.  Returns (X, error word)."""
    lib = _load()
    emb = emb.detach().cpu().contiguous()
    hid = target_hidden.detach().cpu().contiguous()
    hs = h_shared.detach().cpu().contiguous()
    tok = _i32(out_tokens)
    hmap = _i32(hidden_map)
    msk = is_masked.detach().to("cpu", torch.uint8).contiguous()
    T, R = tok.numel(), hmap.numel()
    if X is None:
        X = torch.zeros(T, 2 * H, dtype=emb.dtype)
    else:
        X = X.detach().cpu().contiguous().clone()
    err = ctypes.c_uint32(0)
    _check(lib.oracle_assemble_draft_inputs(
        emb.element_size(), H, V, T, R, _ptr(emb), _ptr(hid), _ptr(hs), _ptr(tok),
        _ptr(hmap), _ptr(msk), _ptr(X), ctypes.byref(err)), "assemble")
    return X, err.value


def step(w) -> dict:
    """The whole step on a workload (see speculative_decoding_pe_gb300.workloads).

    ``w`` carries CPU tensors: logits, in_offsets (prefill) or None, in_tokens,
    in_positions, block_table, emb, hidden, h_shared and the sizes B, Kp, K, V,
    H, mask_id, block_size.  Returns every output plus ``err``."""
    lib = _load()
    B, Kp, K, V, H = w.B, w.Kp, w.K, w.V, w.H
    logits = w.logits.detach().cpu()
    assert logits.stride(1) == 1
    in_offsets = _i32(w.in_offsets)
    R = int(in_offsets[B]) if in_offsets is not None else B * (Kp + 1)
    T = R + B * (K - 1)
    o = _rebuild_outputs(B, K, R, T)
    o["accepted_len"] = torch.full((B,), -7, dtype=torch.int32)
    o["bonus_token"] = torch.full((B,), -7, dtype=torch.int32)
    o["target_argmax"] = torch.full((B * (Kp + 1),), -7, dtype=torch.int32)
    emb = w.emb.detach().cpu().contiguous()
    hid = w.hidden.detach().cpu().contiguous()
    hs = w.h_shared.detach().cpu().contiguous()
    o["X"] = torch.zeros(T, 2 * H, dtype=emb.dtype)
    bt = _i32(w.block_table)
    err = ctypes.c_uint32(0)
    _check(lib.oracle_step(
        _dt(logits), _dt(emb), B, Kp, K, V, H, w.mask_id, _ptr(logits),
        logits.stride(0), _ptr(in_offsets), _ptr(_i32(w.in_tokens)),
        _ptr(_i32(w.in_positions)), _ptr(bt), bt.shape[1], w.block_size,
        _ptr(emb), _ptr(hid), _ptr(hs), _ptr(o["accepted_len"]),
        _ptr(o["bonus_token"]), _ptr(o["target_argmax"]), _ptr(o["out_offsets"]),
        _ptr(o["out_tokens"]), _ptr(o["out_positions"]), _ptr(o["is_rejected"]),
        _ptr(o["is_masked"]), _ptr(o["hidden_map"]), _ptr(o["slot_mapping"]),
        _ptr(o["sample_idx"]), _ptr(o["X"]), ctypes.byref(err)), "step")
    o["err"] = err.value
    return o
