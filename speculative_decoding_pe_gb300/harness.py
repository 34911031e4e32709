"""Glue between a synthetic workload and the fused step: allocate the outputs
with torch, pack the launch arguments once, and launch.  No arithmetic of the
step happens here."""
from __future__ import annotations

import torch

from . import _native


def allocate(w, device="cuda", sample_idx=True, target_argmax=True):
    """Outputs, zeroed workspace and error word for workload ``w``."""
    out = _native.StepOutputs.empty(w.B, w.Kp, w.K, w.R, w.H, w.emb.dtype, device,
                                    sample_idx, target_argmax)
    ws = _native.new_workspace(w.B * (w.Kp + 1), w.B, device)
    err = _native.new_error_word(device)
    return out, ws, err


def pack(w, out, ws, err) -> _native.StepArgs:
    """pe_step arguments for workload ``w`` (tensors already on the GPU)."""
    return _native.make_step_args(
        logits=w.logits, Kp=w.Kp, K=w.K, mask_id=w.mask_id, in_offsets=w.in_offsets,
        in_tokens=w.in_tokens, in_positions=w.in_positions, block_table=w.block_table,
        block_size=w.block_size, emb=w.emb, target_hidden=w.hidden, h_shared=w.h_shared,
        out=out, workspace=ws, err=err)


def run(w, out, ws, err, stream=None, early_exit=False):
    args = pack(w, out, ws, err)
    if early_exit:
        _native.step_early_exit_packed(args, stream)
    else:
        _native.step_packed(args, stream)


OUTPUT_KEYS = ("accepted_len", "bonus_token", "target_argmax", "out_offsets",
               "out_tokens", "out_positions", "is_rejected", "is_masked", "hidden_map",
               "slot_mapping", "sample_idx", "X")


def to_host(out) -> dict:
    return {k: getattr(out, k).cpu() for k in OUTPUT_KEYS if getattr(out, k) is not None}
