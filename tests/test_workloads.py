"""The seeded input generators (CPU, small shapes)."""
import torch

from speculative_decoding_pe_gb300 import workloads as wl


def _small(name, **kw):
    return wl.SPECS[name].with_(V=3001, H=32, **kw)


def test_deterministic_and_seeded():
    a = wl.make_workload(_small("decode_b64", B=5), 3)
    b = wl.make_workload(_small("decode_b64", B=5), 3)
    c = wl.make_workload(_small("decode_b64", B=5), 4)
    for f in ("logits", "in_tokens", "in_positions", "block_table", "emb", "hidden",
              "h_shared", "planted_accept"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert not torch.equal(a.logits, c.logits)


def test_requests_redraw_alone():
    """Request b's rows depend only on (seed, b), not on the batch size."""
    small = wl.make_workload(_small("decode_b256", B=3), 9)
    big = wl.make_workload(_small("decode_b256", B=7), 9)
    n = small.R
    assert torch.equal(small.in_tokens, big.in_tokens[:n])
    assert torch.equal(small.in_positions, big.in_positions[:n])
    assert torch.equal(small.hidden, big.hidden[:n])
    assert torch.equal(small.logits, big.logits[:small.logits_rows])
    assert torch.equal(small.planted_accept, big.planted_accept[:3])


def test_shapes_and_ranges():
    for name in ("tiny", "decode_b1", "decode_b64", "prefill_b8", "decode_b256"):
        spec = wl.SPECS[name] if name == "tiny" else _small(name, B=min(6, wl.SPECS[name].B),
                                                           prompt_hi=60, prompt_lo=1)
        w = wl.make_workload(spec, 1)
        assert w.logits.shape == (w.logits_rows, w.V)
        assert w.hidden.shape == (w.R, w.H) and w.emb.shape == (w.V, w.H)
        assert w.block_table.shape == (w.B, spec.bt_width)
        assert int(w.in_tokens.max()) < w.mask_id, "drafts never the MASK id"
        assert float(w.logits.float().abs().max()) <= wl.PLANT
        # kept positions fit the block table
        top = int(w.in_positions.max()) + w.K - 1
        assert top // w.block_size < spec.bt_width
        if spec.prefill:
            assert w.in_offsets[0] == 0 and int(w.in_offsets[-1]) == w.R
        else:
            assert w.R == w.B * (w.Kp + 1)
            assert int(w.planted_accept.max()) <= w.Kp


def test_forced_and_padded():
    w = wl.make_workload(wl.SPECS["tiny"].with_(B=3, forced=((0, 3), (2, 0)), row_pad=4), 2)
    assert w.planted_accept[0] == 3 and w.planted_accept[2] == 0
    assert w.logits.stride(0) == w.V + 4
    full = w.logits.as_strided((w.logits_rows, w.V + 4), (w.V + 4, 1))
    assert (full[:, w.V:] == 2 * wl.PLANT).all()
    moved = w.to("cpu")
    assert moved.logits.stride(0) == w.V + 4 and torch.equal(moved.logits, w.logits)
