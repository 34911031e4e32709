"""libpe.so builds here, loads, exports every function include/pe_api.h
declares, and rejects bad arguments on the host before touching CUDA.

No call in this file reaches a kernel: every call fails its host-side checks
(fake pointers are never dereferenced on the host), so it runs without a GPU.
"""
import ctypes
import os
import re

import pytest

from speculative_decoding_pe_gb300 import _native, build

HEADER = os.path.join(build.INCLUDE, "pe_api.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pe_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def test_header_parses():
    names = declared_functions()
    assert "pe_step" in names and "pe_verify_greedy" in names
    assert set(names) == set(_native.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_checked_build_exports_the_same_symbols(lib):
    checked = _native.load_checked()
    for name in declared_functions():
        assert hasattr(checked, name), name
    assert checked.pe_workspace_bytes(2048, 256) == lib.pe_workspace_bytes(2048, 256)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        s = lib.pe_status_str(code).decode()
        assert s.startswith("PE_")
    assert lib.pe_status_str(99) == b"unknown pe_status"


def test_workspace_bytes(lib):
    # scheduler words, then the 1024 chunk-key slots of the single pass
    assert lib.pe_workspace_bytes(0, 0) == (8 + 8 * 1024 + 255) // 256 * 256
    n = lib.pe_workspace_bytes(2048, 256)
    assert n >= 8 + 4 * 256 + 8 * 2048 and n % 256 == 0
    assert lib.pe_workspace_bytes(-1, 3) == 0


FAKE = 0x10000          # 16-byte aligned, never dereferenced on the host
MIS = 0x10004           # misaligned


def _step_args(**over):
    a = _native.StepArgs()
    a.B, a.Kp, a.K, a.V, a.H, a.R = 2, 3, 3, 1000, 64, 8
    a.mask_id, a.bt_width, a.block_size = 999, 64, 16
    a.logits_dtype = a.x_dtype = _native.PE_F32
    a.logits_row_stride = 1000
    for f, _ in _native.StepArgs._fields_[12:]:
        setattr(a, f, FAKE)
    a.in_offsets = None
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,status", [
    ({"logits_dtype": 7}, -2),
    ({"x_dtype": 3}, -2),
    ({"K": 0}, -1),
    ({"Kp": 256}, -1),
    ({"K": 257}, -1),
    ({"mask_id": 1000}, -1),
    ({"mask_id": -1}, -1),
    ({"R": 9}, -1),                      # decode needs R = B*(Kp+1)
    ({"in_offsets": FAKE}, -1),          # decode takes no offsets
    ({"Kp": 0, "R": 8}, -1),             # prefill needs offsets
    ({"X": None}, -1),
    ({"workspace": None}, -1),
    ({"logits_row_stride": 999}, -1),
    ({"logits": MIS}, -3),
    ({"X": MIS}, -3),
    ({"logits_row_stride": 1001}, -3),   # 4004 bytes per row
    ({"H": 65}, -3),                     # 260-byte half rows
    ({"block_size": 0}, -1),
    ({"B": -1}, -1),
])
def test_step_rejects_bad_arguments(lib, over, status):
    a = _step_args(**over)
    assert lib.pe_step(ctypes.byref(a), None) == status


def test_step_null_args(lib):
    assert lib.pe_step(None, None) == -1


def test_verify_rejects(lib):
    f = lib.pe_verify_greedy
    ok = dict(logits=FAKE, dtype=1, stride=1000, B=2, Kp=3, V=1000, tok=FAKE, acc=FAKE,
              bon=FAKE, amax=None, ws=FAKE, err=FAKE)

    def call(**o):
        d = dict(ok, **o)
        return f(d["logits"], d["dtype"], d["stride"], d["B"], d["Kp"], d["V"], d["tok"],
                 d["acc"], d["bon"], d["amax"], d["ws"], d["err"], None)
    assert call(dtype=5) == -2
    assert call(Kp=-1) == -1
    assert call(V=0) == -1
    assert call(tok=None) == -1          # drafts needed when Kp > 0
    assert call(ws=None) == -1
    assert call(logits=MIS) == -3
    assert call(stride=1001) == -3       # 2002-byte rows
    assert call(ws=MIS) == -3
    assert call(B=0) == 0                # nothing to do, nothing enqueued


def test_rebuild_rejects(lib):
    f = lib.pe_build_draft_batch

    def call(B=2, Kp=3, K=3, R=8, offs=None, bt_width=64, bs=16, tok=FAKE):
        return f(B, Kp, K, 7, R, offs, tok, FAKE, FAKE, FAKE, FAKE, bt_width, bs,
                 FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None)
    assert call(K=0) == -1
    assert call(R=9) == -1
    assert call(offs=FAKE, R=7) == -1    # segments need >= Kp+1 rows each
    assert call(bt_width=0) == -1
    assert call(bs=0) == -1
    assert call(tok=None) == -1


def test_assemble_rejects(lib):
    f = lib.pe_assemble_draft_inputs

    def call(dt=0, H=64, V=10, T=5, R=3, emb=FAKE, X=FAKE):
        return f(dt, H, V, T, R, emb, FAKE, FAKE, FAKE, FAKE, FAKE, X, FAKE, None)
    assert call(dt=2) == -2
    assert call(H=0) == -1
    assert call(T=-1) == -1
    assert call(T=0, R=0) == 0
    assert call(emb=None) == -1
    assert call(X=MIS) == -3
    assert call(dt=1, H=4) == -3         # 8-byte half rows


def test_tuning_roundtrip(lib):
    before = _native.get_tuning()
    try:
        _native.set_tuning(ctas_per_sm=2, rows_per_unit=8)
        t = _native.get_tuning()
        assert t["ctas_per_sm"] == 2 and t["rows_per_unit"] == 8
        assert t["chunk_batches"] == before["chunk_batches"]
        with pytest.raises(_native.PEError):
            _native.set_tuning(rows_per_unit=17)
        with pytest.raises(_native.PEError):
            _native.set_tuning(queue_order=3)
        _native.set_tuning(queue_order=2)
        assert _native.get_tuning()["queue_order"] == 2
        _native.set_tuning(early_full_read_mb=64)
        assert _native.get_tuning()["early_full_read_mb"] == 64
        _native.set_tuning(early_full_read_mb=-1)  # -1 stores 0: always the early-exit kernel
        assert _native.get_tuning()["early_full_read_mb"] == 0
        with pytest.raises(_native.PEError):
            _native.set_tuning(early_full_read_mb=-2)
        _native.set_tuning(single_pass=-1)
        assert _native.get_tuning()["single_pass"] == -1
        _native.set_tuning(single_pass=1)
        assert _native.get_tuning()["single_pass"] == 1
        with pytest.raises(_native.PEError):
            _native.set_tuning(single_pass=2)
    finally:
        _native.set_tuning(**{k: (v if v or k != "early_full_read_mb" else -1)
                              for k, v in before.items()})


def test_latency_floor_rejects(lib):
    s = ctypes.c_void_p(0)
    assert lib.pe_latency_floor(0, 0, None, 0, None, s) == -1           # no CTA
    assert lib.pe_latency_floor(4, -1, None, 0, None, s) == -1          # negative hops
    assert lib.pe_latency_floor(4, 1, None, 1, ctypes.c_void_p(FAKE), s) == -1  # no chain
    assert lib.pe_latency_floor(4, 1, ctypes.c_void_p(FAKE), 0, ctypes.c_void_p(FAKE), s) == -1
