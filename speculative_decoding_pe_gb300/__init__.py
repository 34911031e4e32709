"""GB300-native per-step data path of P-EAGLE parallel drafting.

Greedy verification, the fused draft-batch rebuild and the drafter input
assembly run in hand-written CUDA kernels for sm_103a behind the C ABI of
``libpe.so`` (``include/pe_api.h``).  This package holds the ctypes binding
(``_native``), the in-tree build (``build``), seeded synthetic workloads
(``workloads``) and the glue the tests and the benchmark share (``harness``).
"""
from ._native import (DraftBatch, PEError, StepArgs, StepOutputs,  # noqa: F401
                      assemble_draft_inputs, build_draft_batch, draft_readout, get_tuning, load,
                      make_step_args, new_error_word, new_workspace, set_tuning, step,
                      step_packed, verify_greedy, workspace_bytes)
