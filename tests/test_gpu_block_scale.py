"""ZYFA_OPT_BLOCK_SCALE: FP8 P scaled per row and 32-key slice by a power of
two before it is rounded to e4m3, and the P V product taken by the
block-scaled MMA, which divides the power of two back out (ZYFA README,
"Kernel design", per-block scaling; "Clock speed and input values": most
probabilities of a long row lie many binades below the row maximum, where
unscaled e4m3 values turn subnormal or zero).

Parity with the float64 oracle under the FP8 tolerances, alone and with the
rounded-P modes; bitwise determinism; and a row structure where the scaling
decides the result: every key but the first lies about 14 binades below the
first, so the unscaled P of those keys (times the kernel's pre-scale) falls below
half the smallest e4m3 subnormal and rounds to zero, while the scaled P keeps
three significant bits."""

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads
from gpu_util import assert_parity, errors, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()
    yield
    assert zf.zyfa_set_option(zf.ZYFA_OPT_BLOCK_SCALE, 0) == zf.ZYFA_OK
    assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, 0) == zf.ZYFA_OK


def _with(fn, block_scale=1, rounded_p=0):
    assert zf.zyfa_set_option(zf.ZYFA_OPT_BLOCK_SCALE, block_scale) == zf.ZYFA_OK
    assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, rounded_p) == zf.ZYFA_OK
    try:
        return fn()
    finally:
        assert zf.zyfa_set_option(zf.ZYFA_OPT_BLOCK_SCALE, 0) == zf.ZYFA_OK
        assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, 0) == zf.ZYFA_OK


@pytest.mark.parametrize("rounded_p", [0, 1, 2])
@pytest.mark.parametrize("d_qk,layout", [(128, "bshd"), (192, "bhsd")])
@pytest.mark.parametrize("values", ["gaussian", "activation"])
def test_block_scale_parity(rounded_p, d_qk, layout, values):
    w = workloads.Workload("block_scale", "fp8", 1, 1100, 4, 2, d_qk=d_qk, d_v=128,
                           layout=layout, values=values, seed=8500 + d_qk + 10 * rounded_p)
    t = workloads.make_inputs(w)
    O, L = _with(lambda: run_gpu(t, w), rounded_p=rounded_p)
    Oref, Lref = run_oracle(t, w)
    assert_parity(O, L, Oref, Lref, "fp8", f"block scale, rounded P {rounded_p}, d{d_qk} {values}")


def test_block_scale_many_items():
    # 2 x 24 heads x 3 query blocks = 144 items on up to 152 CTAs, then a
    # second shape with more items than CTAs so that CTAs run several items.
    for B, S, H in ((2, 700, 24), (3, 1300, 32)):
        w = workloads.Workload("block_scale_items", "fp8", B, S, H, 8, values="activation",
                               seed=8600 + S)
        t = workloads.make_inputs(w)
        O, L = _with(lambda: run_gpu(t, w))
        Oref, Lref = run_oracle(t, w)
        assert_parity(O, L, Oref, Lref, "fp8", f"block scale B{B} S{S} H{H}")


def test_block_scale_deterministic():
    w = workloads.Workload("block_scale_det", "fp8", 1, 3000, 8, 2, values="activation",
                           seed=8700)
    t = workloads.make_inputs(w)
    runs = [_with(lambda: run_gpu(t, w)) for _ in range(3)]
    for O, L in runs[1:]:
        assert np.array_equal(O, runs[0][0]) and np.array_equal(L, runs[0][1])


def _far_tail_inputs(S: int, H: int, seed: int):
    """q along one axis; key 0 scores 14.25-14.6 (scaled units x sqrt(d)) above
    the others, so every other key has p = 0.53-0.69 x 2^-14 relative to key 0;
    v = 0 for key 0 and about 1 elsewhere, so O measures the tail's mass."""
    g = torch.Generator().manual_seed(seed)
    d = 128
    q = torch.zeros((1, S, H, d))
    q[..., 0] = 8.0
    k = torch.zeros((1, S, H, d))
    k[0, 0, :, 0] = 16.0
    # e4m3 codes 22..28 at descale 2^-4: 1.375 .. 1.75
    k[0, 1:, :, 0] = (22 + 2 * torch.randint(0, 4, (S - 1, H), generator=g)).float() / 16.0
    v = 1.0 + 0.25 * torch.randn((1, S, H, d), generator=g)
    v[0, 0] = 0.0
    (q8, qs), (k8, ks), (v8, vs) = (workloads.fp8_quantize_cpu(x) for x in (q, k, v))
    return dict(q=q8, k=k8, v=v8, q_descale=qs, k_descale=ks, v_descale=vs)


def test_block_scale_keeps_far_tail():
    S, H = 4096, 2
    w = workloads.Workload("far_tail", "fp8", 1, S, H, H, seed=8800)
    t = _far_tail_inputs(S, H, w.seed)
    Oref, Lref = run_oracle(t, w)
    # the tail carries up to 13 % of the weight of the last rows
    assert 0.1 < Oref[0, -1].mean() < 0.2
    O0, L0 = run_gpu(t, w)
    O1, L1 = _with(lambda: run_gpu(t, w))
    e0, e1 = errors(O0, L0, Oref, Lref), errors(O1, L1, Oref, Lref)
    print(f"far tail: unscaled max|dO| {e0['max_o']:.3e} mean {e0['mean_o']:.3e}; "
          f"block-scaled max|dO| {e1['max_o']:.3e} mean {e1['mean_o']:.3e}")
    assert_parity(O1, L1, Oref, Lref, "fp8", "block scale, far tail")
    # unscaled, the tail's P rounds to zero: O stays near 0 where it should
    # reach 0.13
    assert e0["max_o"] > 0.1
    assert e1["max_o"] < 0.25 * e0["max_o"] and e1["mean_o"] < 0.25 * e0["mean_o"]


@pytest.mark.parametrize("rounded_p", [1, 2])
def test_block_scale_weights_sum_to_one(rounded_p):
    # v = 1: with the rounded sum as the denominator every output is exactly
    # 1 in BF16 (the scaled values and their sum carry the same powers of two).
    w = workloads.Workload("ones", "fp8", 1, 777, 4, 2, seed=8900)
    q, k, _ = workloads.fp32_inputs(w)
    (q8, qs), (k8, ks) = workloads.fp8_quantize_cpu(4.0 * q), workloads.fp8_quantize_cpu(4.0 * k)
    v = torch.ones((w.B, w.S, w.Hkv, w.d_v)).to(torch.float8_e4m3fn)
    t = dict(q=q8, k=k8, v=v, q_descale=qs, k_descale=ks, v_descale=1.0)
    O, _ = _with(lambda: run_gpu(t, w), rounded_p=rounded_p)
    assert np.array_equal(O, np.ones_like(O))
