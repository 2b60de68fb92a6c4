"""ZYFA_OPT_ROUNDED_P: O divided by the sum of the rounded probabilities that
multiply V on every tile (mode 1), and the LSE from that same sum (mode 2),
as the ZYFA README describes its kernels ("Accuracy": each output stays a
weighted average whose weights sum to one; the FP8 log-sum-exp comes from the
rounded probabilities so that partial results merge consistently).

Parity with the float64 oracle is checked in both modes.  O keeps the stated
tolerances.  In mode 2 the LSE carries the rounding of P: for BF16 P each
value is within half a BF16 step (2^-8 relative) of the exact one, so the
rounded sum is within that relative error of the exact sum and the LSE within
ln(1 + 2^-8) = 3.9e-3 nats; FP8 keeps its stated 5e-3 bound (its dominant
tiles carry the two-term P of about 8 significant bits)."""

import math

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads
from gpu_util import TOL, Tol, assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

LSE_MODE2 = {"bf16": math.log1p(2.0 ** -8) + 1e-4, "fp8": 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()
    yield
    assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, 0) == zf.ZYFA_OK


def _with_mode(mode, fn):
    assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, mode) == zf.ZYFA_OK
    try:
        return fn()
    finally:
        assert zf.zyfa_set_option(zf.ZYFA_OPT_ROUNDED_P, 0) == zf.ZYFA_OK


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("d_qk,layout", [(128, "bshd"), (192, "bhsd")])
@pytest.mark.parametrize("values", ["gaussian", "activation"])
def test_rounded_p_parity(mode, dtype, d_qk, layout, values):
    w = workloads.Workload("rounded_p", dtype, 1, 1100, 4, 2, d_qk=d_qk, d_v=128, layout=layout,
                           values=values, seed=8100 + d_qk + (dtype == "fp8") + 10 * mode)
    t = workloads.make_inputs(w)
    O, L = _with_mode(mode, lambda: run_gpu(t, w))
    Oref, Lref = run_oracle(t, w)
    tol = TOL[dtype]
    if mode == 2:
        tol = Tol(tol.max_o, tol.mean_o, LSE_MODE2[dtype])
    assert_parity(O, L, Oref, Lref, dtype, f"rounded P mode {mode} {dtype} d{d_qk} {values}",
                  tol=tol)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_weights_sum_to_one(dtype):
    # v = 1 everywhere, so O is the sum of each row's weights.  q and k with
    # a large spread make rows where one key dominates (and the rescale, two-
    # term and exact paths all run).  With the rounded sum as denominator
    # every output is exactly 1 in BF16.
    w = workloads.Workload("ones", dtype, 1, 777, 4, 2, seed=8300 + (dtype == "fp8"))
    q, k, _ = workloads.fp32_inputs(w)
    q, k = 4.0 * q, 4.0 * k
    v = torch.ones((w.B, w.S, w.Hkv, w.d_v), dtype=torch.float32)
    if dtype == "bf16":
        t = dict(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16),
                 q_descale=1.0, k_descale=1.0, v_descale=1.0)
    else:
        (q8, qs), (k8, ks) = workloads.fp8_quantize_cpu(q), workloads.fp8_quantize_cpu(k)
        t = dict(q=q8, k=k8, v=v.to(torch.float8_e4m3fn), q_descale=qs, k_descale=ks,
                 v_descale=1.0)
    O1, _ = _with_mode(1, lambda: run_gpu(t, w))
    O0, _ = run_gpu(t, w)
    print(f"{dtype}: default mode max|O-1| = {np.abs(O0 - 1).max():.3e}, "
          f"rounded-P mode max|O-1| = {np.abs(O1 - 1).max():.3e}")
    assert np.array_equal(O1, np.ones_like(O1))
    # The rows are peaked: in most of them one key carries over half the
    # weight (float64 probabilities of head 0 from the oracle).
    import oracle
    Q, K, _ = oracle.decode_inputs_f64(workloads.codes(t["q"]), workloads.codes(t["k"]),
                                       workloads.codes(t["v"]), dtype=dtype, layout=w.layout,
                                       q_descale=t["q_descale"], k_descale=t["k_descale"],
                                       v_descale=t["v_descale"])
    P, _, _ = oracle.causal_probs_f64(Q[0, 0], K[0, 0], 1.0 / math.sqrt(w.d_qk))
    assert np.mean(P.max(axis=1) > 0.5) > 0.5
