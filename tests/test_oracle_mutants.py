"""Plausible mistakes planted in a copy of the oracle must fail a pin.

Each mutant rewrites one expression of ``oracle/pe_oracle.c`` (a dropped
term, a wrong index, an inverted tie rule ...), compiles it with gcc into a
temporary library and runs the pin suite against it.  The real oracle is
never modified; this runs on the CPU only.
"""
import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RUNNER = """
import json, sys
sys.path[:0] = [%r, %r]
import oracle, pins
oracle.use_library(%r)
failed = []
for pin in pins.ALL_PINS:
    try:
        pin()
    except AssertionError:
        failed.append(pin.__name__)
print(json.dumps(failed))
"""

MUTANTS = {
    "argmax_ties_to_last": ("if (x > best_val)", "if (x >= best_val)"),
    "compare_unshifted_draft": ("amax[first + j] != tokens[first + j + 1]",
                                "amax[first + j] != tokens[first + j]"),
    "bonus_from_last_row": ("bonus_token[b] = amax[first + a];",
                            "bonus_token[b] = amax[first + Kp];"),
    "accepted_token_not_shifted": ("if (k < s) { /* accepted / prompt slot: token shifted by one */\n        tok = in_tokens[io[b] + k + 1];",
                                   "if (k < s) { /* accepted / prompt slot: token shifted by one */\n        tok = in_tokens[io[b] + k];"),
    "bonus_slot_ignores_prefill": ("s = n - 1 - Kp + a;", "s = a;"),
    "mask_position_off_by_one": ("pos = in_positions[io[b] + s] + (k - n + 1);",
                                 "pos = in_positions[io[b] + s] + (k - n);"),
    "rejected_filler_always_mask": ("tok = (k < n - 1) ? in_tokens[io[b] + k + 1] : mask_id;",
                                    "tok = mask_id;"),
    "rejected_not_padded": ("if (rej) {\n        slot_mapping[t] = -1;",
                            "if (0) {\n        slot_mapping[t] = -1;"),
    "slot_offset_dropped": ("slot_mapping[t] = blk * block_size + (pos % block_size);",
                            "slot_mapping[t] = blk * block_size;"),
    "offsets_scan_drops_mask_rows": ("oo[b + 1] = oo[b] + (io[b + 1] - io[b]) + (K - 1);",
                                     "oo[b + 1] = oo[b] + (io[b + 1] - io[b]) + (K - 1) / 2;"),
    "hidden_map_shifted": ("hidden_map[io[b] + k] = oo[b] + k;",
                           "hidden_map[io[b] + k] = oo[b] + k + (k > 0);"),
    "sample_idx_skips_first_mask": ("sample_idx[(int64_t)b * K + k] = oo[b] + n + k - 1;",
                                    "sample_idx[(int64_t)b * K + k] = oo[b] + n + k;"),
    "h_shared_not_broadcast": ("if (is_masked[t]) memcpy(",
                               "if (0 && is_masked[t]) memcpy("),
    "emb_of_wrong_row": ("memcpy(dst, (const char*)emb + (size_t)tok * half, half);",
                         "memcpy(dst, (const char*)emb + (size_t)(tok ^ 1) * half, half);"),
    "bf16_low_half": ("bits = ((uint32_t)h) << 16;", "bits = ((uint32_t)h);"),
    "readout_ignores_sample_idx": ("int32_t r = sample_idx ? sample_idx[i] : i;",
                                   "int32_t r = i;"),
    "sampled_accept_ignores_q": ("if (!((double)u_accept[(int64_t)b * Kp + j] * qx < px)) {",
                                 "if (!((double)u_accept[(int64_t)b * Kp + j] < px + 0.0 * qx)) {"),
    "sampled_residual_is_p": ("if (pv - qv > 0.0) {\n          double sc = log(pv - qv)",
                              "if (pv > 0.0 * qv) {\n          double sc = log(pv)"),
    "gumbel_sign_flipped": ("return -log(-log(u));", "return log(-log(u));"),
    "philox_nine_rounds": ("for (r = 0; r < 10; ++r) {", "for (r = 0; r < 9; ++r) {"),
}


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, workdir):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, "mutation site not found exactly once: %s" % name
    path = os.path.join(workdir, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(workdir, name + ".so"))
    # a separate process, so that a mutant that corrupts memory cannot take
    # the test session down with it
    code = RUNNER % (ROOT, os.path.join(ROOT, "tests"), lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, "mutant %s crashed: %s" % (name, res.stderr[-2000:])
    failed = json.loads(res.stdout.strip().splitlines()[-1])
    assert failed, "no pin caught mutant %s" % name
