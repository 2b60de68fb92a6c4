"""The C ABI without a GPU: the library loads, exports every declared symbol,
and its host-side argument checks return the documented status codes before
any CUDA call."""

import math
import os
import re

import pytest

import causal_flashattention_prefill_gb300 as zf
from causal_flashattention_prefill_gb300 import build as zbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return zf.load()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "zyfa.h")).read()
    return re.findall(r"ZYFA_API\s+[\w\s\*]+?\b(zyfa_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = set(_declared_symbols())
    assert {"zyfa_fwd", "zyfa_fwd_scaled", "zyfa_validate", "zyfa_status_string",
            "zyfa_device_status", "zyfa_set_option", "zyfa_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    assert set(_declared_symbols()) <= set(zf._lib.SIGNATURES)


def test_header_enums_match_binding():
    text = open(os.path.join(ROOT, "include", "zyfa.h")).read()
    for name in ("ZYFA_OK", "ZYFA_ERR_ARG", "ZYFA_ERR_UNSUPPORTED", "ZYFA_ERR_ALIGN",
                 "ZYFA_ERR_LAUNCH", "ZYFA_ERR_DEVICE", "ZYFA_ERR_DEVICE_TIMEOUT", "ZYFA_BF16",
                 "ZYFA_FP8_E4M3", "ZYFA_BSHD", "ZYFA_BHSD", "ZYFA_OPT_SERIALIZE_PV",
                 "ZYFA_OPT_ROUNDED_P", "ZYFA_OPT_BLOCK_SCALE",
                 "ZYFA_OPT_DYNAMIC_SCHEDULE"):
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m, name
        assert int(m.group(1)) == getattr(zf, name), name


def test_version_and_status_strings(lib):
    assert zf.zyfa_version() >> 16 == 1
    for st in range(-6, 1):
        s = zf.zyfa_status_string(st)
        assert s and s != "unknown status"
    assert zf.zyfa_status_string(17) == "unknown status"


A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


def _args(**kw):
    a = dict(q=A, k=A, v=A, out=A, lse=A, B=1, S=256, H=4, Hkv=2, d_qk=128, d_v=128,
             dtype=zf.ZYFA_BF16, q_descale=0, k_descale=0, v_descale=0,
             scale=1 / math.sqrt(128), layout=zf.ZYFA_BSHD)
    a.update(kw)
    return a


def _validate(**kw):
    a = _args(**kw)
    return zf.zyfa_validate(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["S"], a["H"],
                            a["Hkv"], a["d_qk"], a["d_v"], a["dtype"], a["q_descale"],
                            a["k_descale"], a["v_descale"], a["scale"], a["layout"])


CASES = [
    ({}, zf.ZYFA_OK),
    (dict(lse=0), zf.ZYFA_OK),
    (dict(layout=zf.ZYFA_BHSD), zf.ZYFA_OK),
    (dict(d_qk=192), zf.ZYFA_OK),
    (dict(S=1), zf.ZYFA_OK),
    (dict(S=30000, B=2, H=32, Hkv=32), zf.ZYFA_OK),
    (dict(H=4, Hkv=1), zf.ZYFA_OK),
    (dict(dtype=zf.ZYFA_FP8_E4M3, q_descale=A, k_descale=A, v_descale=A), zf.ZYFA_OK),
    (dict(q=0), zf.ZYFA_ERR_ARG),
    (dict(out=0), zf.ZYFA_ERR_ARG),
    (dict(B=0), zf.ZYFA_ERR_ARG),
    (dict(S=0), zf.ZYFA_ERR_ARG),
    (dict(S=-5), zf.ZYFA_ERR_ARG),
    (dict(H=6, Hkv=4), zf.ZYFA_ERR_ARG),
    (dict(Hkv=0), zf.ZYFA_ERR_ARG),
    (dict(layout=2), zf.ZYFA_ERR_ARG),
    (dict(scale=0.0), zf.ZYFA_ERR_ARG),
    (dict(scale=-1.0), zf.ZYFA_ERR_ARG),
    (dict(scale=float("nan")), zf.ZYFA_ERR_ARG),
    (dict(scale=float("inf")), zf.ZYFA_ERR_ARG),
    (dict(d_qk=64, d_v=64), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(d_qk=192, d_v=192), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(d_qk=256), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(dtype=2), zf.ZYFA_ERR_UNSUPPORTED),        # e.g. FP16: not supported
    (dict(dtype=zf.ZYFA_FP8_E4M3), zf.ZYFA_ERR_ARG),  # FP8 without descales
    (dict(dtype=zf.ZYFA_FP8_E4M3, q_descale=A, k_descale=A, v_descale=A + 2), zf.ZYFA_ERR_ALIGN),
    (dict(q=A + 8), zf.ZYFA_ERR_ALIGN),
    (dict(v=A + 2), zf.ZYFA_ERR_ALIGN),
    (dict(out=A + 4), zf.ZYFA_ERR_ALIGN),
    (dict(lse=A + 2), zf.ZYFA_ERR_ALIGN),
    (dict(B=2 ** 20, H=2 ** 10, S=2 ** 20), zf.ZYFA_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("kw,expected", CASES, ids=[str(c[0]) or "valid" for c in CASES])
def test_validation(lib, kw, expected):
    assert _validate(**kw) == expected


@pytest.mark.parametrize("kw,expected", [c for c in CASES if c[1] != zf.ZYFA_OK])
def test_fwd_rejects_before_any_cuda_call(lib, kw, expected):
    """Invalid arguments return their status from zyfa_fwd_scaled without a GPU."""
    a = _args(**kw)
    st = zf.zyfa_fwd_scaled(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["S"], a["H"],
                            a["Hkv"], a["d_qk"], a["d_v"], a["dtype"], a["q_descale"],
                            a["k_descale"], a["v_descale"], a["scale"], a["layout"], 0)
    assert st == expected


def test_options(lib):
    assert zf.zyfa_set_option(zf.ZYFA_OPT_SERIALIZE_PV, 1) == zf.ZYFA_OK
    assert zf.zyfa_set_option(zf.ZYFA_OPT_SERIALIZE_PV, 0) == zf.ZYFA_OK
    for mode in (1, 2, 0):
        assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, mode) == zf.ZYFA_OK
    assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, 3) == zf.ZYFA_ERR_ARG
    assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, -1) == zf.ZYFA_ERR_ARG
    for v in (1, 0):
        assert zf.zyfa_set_option(zf.ZYFA_OPT_BLOCK_SCALE, v) == zf.ZYFA_OK
    assert zf.zyfa_set_option(zf.ZYFA_OPT_BLOCK_SCALE, 2) == zf.ZYFA_ERR_ARG
    assert zf.zyfa_set_option(zf.ZYFA_OPT_BLOCK_SCALE, -1) == zf.ZYFA_ERR_ARG
    for v in (1, 0):
        assert zf.zyfa_set_option(zf.ZYFA_OPT_DYNAMIC_SCHEDULE, v) == zf.ZYFA_OK
    assert zf.zyfa_set_option(zf.ZYFA_OPT_DYNAMIC_SCHEDULE, 2) == zf.ZYFA_ERR_ARG
    assert zf.zyfa_set_option(99, 1) == zf.ZYFA_ERR_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(zf._lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        zf._lib.load(str(tmp_path / "missing.so"))


QUANT_CASES = [
    (dict(x=0), zf.ZYFA_ERR_ARG),
    (dict(x8=0), zf.ZYFA_ERR_ARG),
    (dict(descale=0), zf.ZYFA_ERR_ARG),
    (dict(ws=0), zf.ZYFA_ERR_ARG),
    (dict(n=-1), zf.ZYFA_ERR_ARG),
    (dict(dt=zf.ZYFA_FP8_E4M3), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(dt=7), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(x=A + 8), zf.ZYFA_ERR_ALIGN),
    (dict(x8=A + 4), zf.ZYFA_ERR_ALIGN),
    (dict(descale=A + 2), zf.ZYFA_ERR_ALIGN),
]


@pytest.mark.parametrize("kw,expected", QUANT_CASES, ids=[str(c[0]) for c in QUANT_CASES])
def test_quantize_rejects_before_any_cuda_call(lib, kw, expected):
    a = dict(x=A, n=1024, dt=zf.ZYFA_BF16, x8=A, descale=A, ws=A)
    a.update(kw)
    assert zf.zyfa_fp8_quantize(a["x"], a["n"], a["dt"], a["x8"], a["descale"], a["ws"], 0) == expected


def test_quantize_workspace_size(lib):
    assert zf.zyfa_fp8_quantize_workspace_bytes() == 4096


ROT_CASES = [
    (dict(x=0), zf.ZYFA_ERR_ARG),
    (dict(signs=0), zf.ZYFA_ERR_ARG),
    (dict(x8=0), zf.ZYFA_ERR_ARG),
    (dict(descale=0), zf.ZYFA_ERR_ARG),
    (dict(ws=0), zf.ZYFA_ERR_ARG),
    (dict(rows=-1), zf.ZYFA_ERR_ARG),
    (dict(rows=1 << 40), zf.ZYFA_ERR_ARG),
    (dict(rows=1 << 31), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(d=64), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(d=256), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(dt=zf.ZYFA_FP8_E4M3), zf.ZYFA_ERR_UNSUPPORTED),
    (dict(x=A + 8), zf.ZYFA_ERR_ALIGN),
    (dict(x8=A + 4), zf.ZYFA_ERR_ALIGN),
    (dict(x8=A + 8), zf.ZYFA_ERR_ALIGN),   # codes are written as 16-byte chunks
    (dict(signs=A + 2), zf.ZYFA_ERR_ALIGN),
]


@pytest.mark.parametrize("kw,expected", ROT_CASES, ids=[str(c[0]) for c in ROT_CASES])
def test_rotated_quantize_rejects_before_any_cuda_call(lib, kw, expected):
    a = dict(x=A, rows=64, d=128, dt=zf.ZYFA_BF16, signs=A, x8=A, descale=A, ws=A)
    a.update(kw)
    assert zf.zyfa_fp8_quantize_rotated(a["x"], a["rows"], a["d"], a["dt"], a["signs"], a["x8"],
                                        a["descale"], a["ws"], 0) == expected
