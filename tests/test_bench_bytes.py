"""The roofline numerator: bench.algorithmic_bytes against the byte counts of
the step written out by hand for each workload (every byte read or written
once: logits rows, target hidden rows, one embedding row per verified or
prompt slot plus the MASK row, X written once, the metadata vectors)."""
import pytest

import bench
from speculative_decoding_pe_gb300 import workloads as wl

# (workload, B, K', K, H, V, element bytes, expected total), totals rounded as
# quoted: tiny 85.5 KB, B=1 3.48 MB, B=64 222.2 MB, B=256 668.6 MB.
CASES = [("tiny", 4, 3, 3, 64, 1000, 4, 85.5e3),
         ("decode_b1", 1, 7, 7, 2880, 201088, 2, 3.48e6),
         ("decode_b64", 64, 7, 7, 2880, 201088, 2, 222.2e6),
         ("decode_b256", 256, 7, 7, 2048, 151936, 2, 668.6e6)]


@pytest.mark.parametrize("name,B,Kp,K,H,V,elt,total", CASES, ids=[c[0] for c in CASES])
def test_decode_bytes(name, B, Kp, K, H, V, elt, total):
    spec = wl.SPECS[name]
    assert (spec.B, spec.Kp, spec.K, spec.H, spec.V) == (B, Kp, K, H, V)
    R = B * (Kp + 1)
    got = bench.algorithmic_bytes(spec, R)
    assert got["logits"] == R * V * elt
    assert got["hidden"] == R * H * elt
    assert got["emb"] == (R + 1) * H * elt
    assert got["X"] == (R + B * (K - 1)) * 2 * H * elt
    assert got["total"] == sum(v for k, v in got.items() if k != "total")
    assert abs(got["total"] - total) / total < 0.002, got["total"]


def test_prefill_bytes():
    """First step after prefill, B=8 prompts of the expected total length
    36864 tokens: about 854 MB, dominated by hidden rows read and X written."""
    spec = wl.SPECS["prefill_b8"]
    R = 36864
    got = bench.algorithmic_bytes(spec, R)
    assert got["logits"] == 8 * 201088 * 2  # the last row of each prompt
    assert got["hidden"] == R * 2880 * 2
    assert got["X"] == (R + 8 * 6) * 2 * 2880 * 2
    assert abs(got["total"] - 854.2e6) / 854.2e6 < 0.002, got["total"]


def test_early_exit_counts_needed_rows_only():
    spec = wl.SPECS["decode_b256"]
    full = bench.algorithmic_bytes(spec, 2048)
    early = bench.algorithmic_bytes(spec, 2048, logits_rows=729)
    assert full["logits"] - early["logits"] == (2048 - 729) * 151936 * 2
    assert early["hidden"] == full["hidden"] and early["X"] == full["X"]


def test_sampled_bytes():
    """Rejection sampling at B=256, K'=7, V=151936 bf16 with 141 requests
    rejecting a draft: 3840 rows read once (1.1670 GB) plus the target and
    draft row of each rejection again (85.7 MB): 1.253 GB with the tokens,
    coins and outputs."""
    got = bench.sampled_bytes(256, 7, 151936, 2, 141)
    assert got["logits"] == (256 * 8 + 256 * 7) * 151936 * 2
    assert got["residual_reread"] == 141 * 2 * 151936 * 2
    assert abs(got["total"] - 1.2526e9) / 1.2526e9 < 0.001, got["total"]
