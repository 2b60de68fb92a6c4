"""ZYFA_OPT_DYNAMIC_SCHEDULE: work items go to whichever SM frees up first
(one CTA per item; running CTAs take the items of CTAs that have not started)
instead of the static deal over one persistent CTA per SM (ZYFA README,
"Kernel design": longest-first work distribution).

Every item is computed the same way wherever it runs, so the outputs must be
bitwise identical to the static schedule's; they are also compared with the
oracle, on shapes with fewer items than SMs, a few rounds of items, and many
rounds, for both input types and head-dim forms."""

import numpy as np
import pytest

import causal_flashattention_prefill_gb300 as zf
import workloads
from gpu_util import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()
    yield
    assert zf.zyfa_set_option(zf.ZYFA_OPT_DYNAMIC_SCHEDULE, 0) == zf.ZYFA_OK


def _dynamic(fn):
    assert zf.zyfa_set_option(zf.ZYFA_OPT_DYNAMIC_SCHEDULE, 1) == zf.ZYFA_OK
    try:
        return fn()
    finally:
        assert zf.zyfa_set_option(zf.ZYFA_OPT_DYNAMIC_SCHEDULE, 0) == zf.ZYFA_OK


CASES = [
    # (dtype, B, S, H, Hkv, d_qk, layout, values): 8, 144, 312 and 2048 items
    ("bf16", 1, 1000, 2, 1, 128, "bshd", "gaussian"),
    ("fp8", 2, 700, 24, 8, 128, "bshd", "activation"),
    ("bf16", 3, 1300, 32, 8, 128, "bhsd", "gaussian"),
    ("fp8", 1, 1300, 24, 24, 192, "bhsd", "activation"),
    ("bf16", 2, 2000, 16, 16, 192, "bhsd", "gaussian"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}S{c[2]}H{c[3]}-d{c[5]}")
def test_dynamic_equals_static_and_oracle(case):
    dtype, B, S, H, Hkv, d_qk, layout, values = case
    w = workloads.Workload("schedule", dtype, B, S, H, Hkv, d_qk=d_qk, d_v=128, layout=layout,
                           values=values, seed=9100 + S + H)
    t = workloads.make_inputs(w)
    O_static, L_static = run_gpu(t, w)
    O_dyn, L_dyn = _dynamic(lambda: run_gpu(t, w))
    assert np.array_equal(O_dyn, O_static) and np.array_equal(L_dyn, L_static)
    Oref, Lref = run_oracle(t, w)
    assert_parity(O_dyn, L_dyn, Oref, Lref, dtype, f"dynamic schedule {case}")


def test_dynamic_full_size_bitwise():
    # The S = 16384 GQA shape: 2048 items, about 13 per SM (compared on the
    # device).
    import torch
    from gpu_util import device_inputs
    w = workloads.WORKLOADS["fp8_gqa_b1_h32kv8_s16384_d128"]
    t = workloads.make_inputs(w)
    q, k, v, ds = device_inputs(t, w)

    def call():
        o, lse = zf.attention(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2],
                              layout=w.layout, return_lse=True)
        torch.cuda.synchronize()
        return o, lse

    O_static, L_static = call()
    for _ in range(2):
        O, L = _dynamic(call)
        assert torch.equal(O, O_static) and torch.equal(L, L_static)
