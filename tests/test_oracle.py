"""Pins of the float64 oracle against facts that do not come from the oracle.

Each ``pin_*`` checks the oracle against something independent of it: a
hand-worked example, closed forms, invariants of the definition, brute force
on tiny inputs, or a library routine for the special case.  ``test_mutants``
plants plausible mistakes in the oracle (on the CPU) and checks that at least
one pin catches each of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as oa
from oracle.formats import bf16_to_f64, e4m3_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _attn(Q, K, V, scale=None):
    """Oracle on float64 (B,H,S,d) inputs, returning O (B,H,S,dv) and LSE."""
    return oracle.attention_f64(Q, K, V, dtype="f64", layout="bhsd", scale=scale)


# ----------------------------------------------------------------- the pins

def pin_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_s3.json")))
    Q = np.array(g["q"])[None, None]
    K = np.array(g["k"])[None, None]
    V = np.array(g["v"])[None, None]
    O, L = _attn(Q, K, V, scale=g["scale"])
    np.testing.assert_allclose(O[0, 0], np.array(g["O"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], np.array(g["LSE"]), rtol=0, atol=1e-14)


def pin_row0_is_v0():
    B, H, Hkv, S, d = 2, 4, 2, 9, 16
    Q, K, V = _rand((B, H, S, d), 1), _rand((B, Hkv, S, d), 2), _rand((B, Hkv, S, d), 3)
    O, L = _attn(Q, K, V)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            assert np.array_equal(O[b, h, 0], V[b, hk, 0])
            assert abs(L[b, h, 0] - Q[b, h, 0] @ K[b, hk, 0] / math.sqrt(d)) < 1e-13


def pin_probs_sum_to_one():
    S, d = 33, 8
    Q, K = _rand((S, d), 4, 3.0), _rand((S, d), 5, 3.0)
    P, m, l = oa.causal_probs_f64(Q, K, 1.0 / math.sqrt(d))
    assert np.all(np.abs(P.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(P[np.triu_indices(S, 1)] == 0.0)
    assert np.all(P[np.tril_indices(S)] > 0.0)


def pin_lse_bruteforce():
    B, H, S, d = 1, 2, 20, 8
    Q, K, V = _rand((B, H, S, d), 6), _rand((B, H, S, d), 7), _rand((B, H, S, d), 8)
    scale = 0.3
    _, L = _attn(Q, K, V, scale=scale)
    for h in range(H):
        for i in range(S):
            s = sum(math.exp(scale * float(np.dot(Q[0, h, i], K[0, h, j])))
                    for j in range(i + 1))
            assert abs(L[0, h, i] - math.log(s)) <= 1e-12


def pin_q_zero_closed_form():
    B, H, S, d = 1, 3, 40, 8
    Q = np.zeros((B, H, S, d))
    K, V = _rand((B, H, S, d), 9), _rand((B, H, S, d), 10)
    O, L = _attn(Q, K, V)
    cummean = np.cumsum(V, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    np.testing.assert_allclose(O, cummean, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, np.log(np.arange(1, S + 1))[None, None, :]
                               * np.ones((B, H, 1)), rtol=0, atol=1e-13)


def pin_constant_v():
    B, H, S, d = 1, 2, 25, 8
    Q, K = _rand((B, H, S, d), 11, 4.0), _rand((B, H, S, d), 12, 4.0)
    V = np.full((B, H, S, d), -1.75)
    O, _ = _attn(Q, K, V)
    np.testing.assert_allclose(O, V, rtol=0, atol=1e-13)


def pin_gqa_is_mha_with_repeated_kv():
    B, H, Hkv, S, d = 2, 8, 2, 17, 16
    Q, K, V = _rand((B, H, S, d), 13), _rand((B, Hkv, S, d), 14), _rand((B, Hkv, S, d), 15)
    O1, L1 = _attn(Q, K, V)
    rep = H // Hkv
    O2, L2 = _attn(Q, np.repeat(K, rep, axis=1), np.repeat(V, rep, axis=1))
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-13)


def pin_zero_padding_leaves_real_rows():
    B, H, S, Sp, d = 1, 2, 37, 64, 16
    Q, K, V = _rand((B, H, S, d), 16), _rand((B, H, S, d), 17), _rand((B, H, S, d), 18)
    pad = lambda t: np.concatenate([t, np.zeros((B, H, Sp - S, d))], axis=2)  # noqa: E731
    O1, L1 = _attn(Q, K, V)
    O2, L2 = _attn(pad(Q), pad(K), pad(V))
    np.testing.assert_allclose(O2[:, :, :S], O1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2[:, :, :S], L1, rtol=0, atol=1e-12)


def _scalar_attention(Q, K, V, scale):
    """Pure-Python triple loop, no numpy arithmetic (independent restatement)."""
    S, dv = len(Q), len(V[0])
    O, L = [], []
    for i in range(S):
        s = [scale * sum(Q[i][c] * K[j][c] for c in range(len(Q[i])))
             for j in range(i + 1)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        O.append([sum(e[j] * V[j][c] for j in range(i + 1)) / tot for c in range(dv)])
        L.append(m + math.log(tot))
    return O, L


def pin_scalar_triple_loop():
    B, H, Hkv, S, dqk, dv = 1, 4, 2, 12, 6, 5
    Q, K, V = _rand((B, H, S, dqk), 19, 2.0), _rand((B, Hkv, S, dqk), 20, 2.0), _rand((B, Hkv, S, dv), 21)
    scale = 1.0 / math.sqrt(dqk)
    O, L = _attn(Q, K, V)
    for h in range(H):
        hk = h // (H // Hkv)
        Os, Ls = _scalar_attention(Q[0, h].tolist(), K[0, hk].tolist(), V[0, hk].tolist(), scale)
        np.testing.assert_allclose(O[0, h], np.array(Os), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[0, h], np.array(Ls), rtol=0, atol=1e-12)


def pin_torch_sdpa_float64():
    B, H, Hkv, S, d = 2, 4, 1, 50, 32
    Q, K, V = _rand((B, H, S, d), 22), _rand((B, Hkv, S, d), 23), _rand((B, Hkv, S, d), 24)
    O, _ = _attn(Q, K, V)
    tq = torch.from_numpy(Q)
    tk = torch.from_numpy(K).repeat_interleave(H // Hkv, dim=1)
    tv = torch.from_numpy(V).repeat_interleave(H // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


def pin_layouts_agree():
    B, H, S, d = 2, 3, 21, 8
    Q, K, V = _rand((B, H, S, d), 25), _rand((B, H, S, d), 26), _rand((B, H, S, d), 27)
    O1, L1 = oracle.attention_f64(Q, K, V, dtype="f64", layout="bhsd")
    t = lambda x: np.transpose(x, (0, 2, 1, 3))  # noqa: E731
    O2, L2 = oracle.attention_f64(t(Q), t(K), t(V), dtype="f64", layout="bshd")
    assert O2.shape == (B, S, H, d)
    np.testing.assert_allclose(t(O2), O1, rtol=0, atol=0)
    np.testing.assert_allclose(L2, L1, rtol=0, atol=0)


def pin_rows_match_full():
    B, H, S, d = 1, 2, 30, 8
    Q, K, V = _rand((B, H, S, d), 28), _rand((B, H, S, d), 29), _rand((B, H, S, d), 30)
    O, L = _attn(Q, K, V)
    rows = np.array([0, 5, 17, 29])
    Or, Lr = oracle.attention_rows_f64(Q, K, V, rows, dtype="f64", layout="bhsd")
    np.testing.assert_allclose(Or, O[:, :, rows], rtol=0, atol=1e-14)
    np.testing.assert_allclose(Lr, L[:, :, rows], rtol=0, atol=1e-14)


PINS = [pin_worked_example, pin_row0_is_v0, pin_probs_sum_to_one,
        pin_lse_bruteforce, pin_q_zero_closed_form, pin_constant_v,
        pin_gqa_is_mha_with_repeated_kv, pin_zero_padding_leaves_real_rows,
        pin_scalar_triple_loop, pin_torch_sdpa_float64, pin_layouts_agree,
        pin_rows_match_full]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# ------------------------------------------------------- planted mistakes

_orig_probs = oa.causal_probs_f64


def _mut_mask_flipped(Qbh, Kbh, scale, rows=None):
    S = Kbh.shape[0]
    rows = np.arange(Qbh.shape[0]) if rows is None else np.asarray(rows)
    sc = scale * (Qbh[rows] @ Kbh.T)
    sc = np.where(np.arange(S)[None, :] >= rows[:, None], sc, -np.inf)
    m = sc.max(axis=1)
    e = np.exp(sc - m[:, None])
    return e / e.sum(axis=1)[:, None], m, e.sum(axis=1)


def _mut_transposed(Qbh, Kbh, scale, rows=None):
    S = Kbh.shape[0]
    rows = np.arange(Qbh.shape[0]) if rows is None else np.asarray(rows)
    sc = scale * (Kbh @ Qbh.T)[rows]
    sc = np.where(np.arange(S)[None, :] <= rows[:, None], sc, -np.inf)
    m = sc.max(axis=1)
    e = np.exp(sc - m[:, None])
    return e / e.sum(axis=1)[:, None], m, e.sum(axis=1)


MUTANTS = {
    "mask_flipped": ("causal_probs_f64", _mut_mask_flipped),
    "transposed_scores": ("causal_probs_f64", _mut_transposed),
    "scale_dropped": ("causal_probs_f64",
                      lambda Q, K, scale, rows=None: _orig_probs(Q, K, 1.0, rows)),
    "max_dropped_from_lse": ("causal_probs_f64",
                             lambda Q, K, scale, rows=None: (
                                 lambda r: (r[0], 0.0 * r[1], r[2]))(_orig_probs(Q, K, scale, rows))),
    "not_normalised": ("causal_probs_f64",
                       lambda Q, K, scale, rows=None: (
                           lambda r: (r[0] * r[2][:, None], r[1], r[2]))(_orig_probs(Q, K, scale, rows))),
    "gqa_modulo_mapping": ("_kv_head", lambda h, H, Hkv: h % Hkv),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(oa, attr, fn)
    caught = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"


# --------------------------------------------------------- input formats

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.isnan(ours).sum() == 2


def test_e4m3_format_facts():
    facts = json.load(open(os.path.join(GOLDEN, "e4m3_format_facts.json")))["facts"]
    vals = e4m3_to_f64(np.arange(128, dtype=np.uint8))     # positive codes
    finite = vals[~np.isnan(vals)]
    assert finite.max() == facts["max_finite"]["value"]
    normals = finite[finite >= facts["min_normal"]["value"]]
    assert normals.min() == facts["min_normal"]["value"]
    # codes 0x08.. are the normals: exponent field >= 1
    assert vals[8] == facts["min_normal"]["value"] and vals[7] < vals[8]
    # the smallest subnormal is 2^-9, so values below 2^-10 round to zero
    assert finite[finite > 0].min() == 2 * facts["round_to_zero_below"]["value"]
    # value doubles every 8 codes among the normals (lean-P relation)
    step = facts["code_step_per_doubling"]["value"]
    for c in range(8, 127 - step):
        assert vals[c + step] == 2 * vals[c]
    assert 1 + facts["exponent_bits"]["value"] + facts["mantissa_bits"]["value"] == 8


def test_bf16_decode_matches_torch():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    ours = bf16_to_f64(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(ours, x.to(torch.float64).numpy())
    special = np.array([0x0000, 0x8000, 0x3F80, 0x7F7F, 0x0001], dtype=np.uint16)
    vals = bf16_to_f64(special)
    assert vals[0] == 0.0 and vals[2] == 1.0 and vals[4] == 2.0 ** -133
    assert vals[3] == (2 - 2 ** -7) * 2.0 ** 127


def test_fp8_inputs_decode_exactly():
    """Oracle decode of quantised inputs equals torch's e4m3 value x descale."""
    import workloads
    w = workloads.WORKLOADS["fp8_gqa_b1_h32kv8_s16384_d128"].with_(S=64)
    t = workloads.make_inputs(w)
    for name in ("q", "k", "v"):
        ref = t[name].to(torch.float64).numpy() * t[name + "_descale"]
        ours = e4m3_to_f64(workloads.codes(t[name]), t[name + "_descale"])
        assert np.array_equal(ours, ref)


# ------------------------------------------------------------- quantiser

from oracle.quantize import descale_of, e4m3_encode_rne, fp8_quantize_f64  # noqa: E402


def test_quantize_encoder_matches_torch():
    """Round-to-nearest-even e4m3 encoding against torch's float8_e4m3fn cast."""
    rng = np.random.default_rng(11)
    y = np.concatenate([
        rng.standard_normal(20000) * 50.0,
        rng.uniform(-448, 448, 20000),
        rng.uniform(-2.0 ** -6, 2.0 ** -6, 20000),        # subnormal range
        e4m3_to_f64(np.arange(0, 126, dtype=np.uint8)),   # exact values
    ]).astype(np.float32).astype(np.float64)
    vals = e4m3_to_f64(np.arange(0, 127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2.0                   # exact ties
    y = np.concatenate([y, mids, -mids])
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode_rne(y), ref)


def test_quantize_ties_and_saturation():
    assert e4m3_encode_rne(np.array([1.0625]))[0] == 0x38      # tie 1.0 | 1.125 -> even
    assert e4m3_encode_rne(np.array([1.1875]))[0] == 0x3A      # tie 1.125 | 1.25 -> even
    assert e4m3_encode_rne(np.array([2.0 ** -10]))[0] == 0x00  # half the smallest subnormal
    assert e4m3_encode_rne(np.array([1000.0]))[0] == 0x7E      # saturates to 448
    assert e4m3_encode_rne(np.array([-1000.0]))[0] == 0xFE


def test_quantize_descale_rule():
    assert descale_of(448.0) == 1.0
    assert descale_of(449.0) == 2.0
    assert descale_of(224.0) == 0.5
    assert descale_of(224.00001) == 1.0
    assert descale_of(0.0) == 1.0
    assert descale_of(3.0) == 2.0 ** -7          # 3 / 2^-7 = 384 <= 448 < 768
    x = np.random.default_rng(3).standard_normal(1000) * 7.0
    codes, d = fp8_quantize_f64(x)
    assert np.abs(x).max() / d <= 448.0 < 2 * np.abs(x).max() / d
    back = e4m3_to_f64(codes) * d
    assert np.all(np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * d))


# ------------------------------------------------------------- rotation

import oracle.rotation as orot  # noqa: E402


def _signs(d, seed):
    return np.where(np.random.default_rng(seed).integers(0, 2, d) == 1, 1.0, -1.0)


def rpin_hadamard_small_cases():
    """Sylvester's construction: H_2 and H_4 written out, H H^T = n I."""
    assert np.array_equal(orot.hadamard_f64(1), [[1.0]])
    assert np.array_equal(orot.hadamard_f64(2), [[1, 1], [1, -1]])
    assert np.array_equal(orot.hadamard_f64(4), [[1, 1, 1, 1], [1, -1, 1, -1],
                                                 [1, 1, -1, -1], [1, -1, -1, 1]])
    for n in (8, 64, 128):
        h = orot.hadamard_f64(n)
        assert np.all(np.abs(h) == 1.0)
        assert np.array_equal(h @ h.T, n * np.eye(n))


def rpin_dct3_closed_form():
    """Orthonormal DCT-II of size 3: rows [1,1,1]/sqrt3, [1,0,-1]/sqrt2, [1,-2,1]/sqrt6."""
    c = orot.dct3_f64()
    want = np.array([[1, 1, 1] / np.sqrt(3), [1, 0, -1] / np.sqrt(2), [1, -2, 1] / np.sqrt(6)])
    np.testing.assert_allclose(c, want, rtol=0, atol=1e-15)
    np.testing.assert_allclose(c @ c.T, np.eye(3), rtol=0, atol=1e-15)


def rpin_orthogonal_and_products_kept():
    """R R^T = I, and (qR)(kR)^T = q k^T: the scores are unchanged."""
    for d in (128, 192):
        s = _signs(d, d)
        r = orot.rotation_f64(d, s)
        np.testing.assert_allclose(r @ r.T, np.eye(d), rtol=0, atol=1e-13)
        q, k = _rand((40, d), 1), _rand((50, d), 2)
        np.testing.assert_allclose(orot.rotate_f64(q, s) @ orot.rotate_f64(k, s).T, q @ k.T,
                                   rtol=0, atol=1e-11)


def rpin_elementwise_definition():
    """Every entry from its definition by plain loops: d=128 R[i,j] =
    s_i H[i,j] / sqrt(128) with H[i,j] = (-1)^popcount(i & j) (the closed
    form of Sylvester's matrix); d=192 R[64a+b, 64c+e] = s_(64a+b) *
    C3[c,a] * (-1)^popcount(b & e) / 8."""
    s = _signs(128, 5)
    r = orot.rotation_f64(128, s)
    for i in range(0, 128, 7):
        for j in range(128):
            want = s[i] * (-1.0) ** bin(i & j).count("1") / math.sqrt(128)
            assert abs(r[i, j] - want) < 1e-15
    s = _signs(192, 6)
    r = orot.rotation_f64(192, s)
    c3 = orot.dct3_f64()
    for a in range(3):
        for b in range(0, 64, 5):
            for cc in range(3):
                for e in range(64):
                    want = s[64 * a + b] * c3[cc, a] * (-1.0) ** bin(b & e).count("1") / 8.0
                    assert abs(r[64 * a + b, 64 * cc + e] - want) < 1e-15


def rpin_unit_vectors():
    """x = e_i gives row i of R, and rotating a quantised tensor is the
    quantisation of x @ R."""
    s = _signs(128, 7)
    r = orot.rotation_f64(128, s)
    np.testing.assert_array_equal(orot.rotate_f64(np.eye(128)[[3, 77]], s), r[[3, 77]])
    x = _rand((9, 128), 8) * 30.0
    codes, d = orot.fp8_quantize_rotated_f64(x, s)
    c2, d2 = fp8_quantize_f64(x @ r)
    assert d == d2 and np.array_equal(codes, c2)


RPINS = [rpin_hadamard_small_cases, rpin_dct3_closed_form, rpin_orthogonal_and_products_kept,
         rpin_elementwise_definition, rpin_unit_vectors]


@pytest.mark.parametrize("pin", RPINS, ids=lambda p: p.__name__)
def test_rotation_pin(pin):
    pin()


_orig_hadamard = orot.hadamard_f64
_orig_dct3 = orot.dct3_f64

ROT_MUTANTS = {
    # H_2n built as [[H, H], [-H, H]] (a plausible sign slip)
    "hadamard_sign_slip": ("hadamard_f64", lambda n: (lambda h: np.block(
        [[h, h], [-h, h]]))(_orig_hadamard(n // 2)) if n > 1 else _orig_hadamard(n)),
    "dct_transposed": ("dct3_f64", lambda: _orig_dct3().T),
    "dct_unnormalised": ("dct3_f64", lambda: _orig_dct3() * math.sqrt(3 / 2)),
}


@pytest.mark.parametrize("name", sorted(ROT_MUTANTS))
def test_rotation_mutants_are_caught(name, monkeypatch):
    attr, fn = ROT_MUTANTS[name]
    monkeypatch.setattr(orot, attr, fn)
    caught = []
    for pin in RPINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every rotation pin"


def test_rotation_mutant_signs_dropped(monkeypatch):
    """Signs ignored: the element-wise pin catches it."""
    orig = orot.rotation_f64
    monkeypatch.setattr(orot, "rotation_f64", lambda d, s: orig(d, np.ones(d)))
    with pytest.raises(AssertionError):
        rpin_elementwise_definition()
