"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Small problems compare every output element; the shape sweep crosses tile
boundaries, ragged tails, GQA/MQA ratios, both layouts, both input formats
and both head-dim forms.  Bitwise properties (run-to-run determinism, layout
and GQA equivalence, the serialized-PV verification mode) compare the CUDA
path with itself.
"""

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads
from gpu_util import assert_parity, run_gpu, run_oracle, to_bhsd

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()
    torch.cuda.init()
    st, v = zf.zyfa_device_status(reset=True)
    assert st == 0


def _check_status():
    st, v = zf.zyfa_device_status()
    assert st == 0 and v == 0, f"device status word {v}"


def test_bf16_b1_h2_s256_full():
    w = W["bf16_mha_b1_h2_s256_d128"]
    t = workloads.make_inputs(w)
    O, L = run_gpu(t, w)
    Oref, Lref = run_oracle(t, w)
    assert_parity(O, L, Oref, Lref, "bf16", w.name)
    _check_status()


def _sweep_cases():
    cases = []
    shapes = [(1, 1, 1), (2, 4, 1), (1, 8, 2), (2, 2, 2), (1, 4, 4)]  # (B, H, Hkv)
    for i, S in enumerate([1, 2, 127, 128, 129, 255, 256, 257, 383, 512, 1000]):
        B, H, Hkv = shapes[i % len(shapes)]
        for dt in ("bf16", "fp8"):
            for d_qk in (128, 192):
                for layout in ("bshd", "bhsd"):
                    cases.append((dt, d_qk, layout, B, S, H, Hkv))
    return cases


@pytest.mark.parametrize("dt,d_qk,layout,B,S,H,Hkv", _sweep_cases(),
                         ids=lambda x: str(x))
def test_shape_sweep(dt, d_qk, layout, B, S, H, Hkv):
    w = workloads.Workload("sweep", dt, B, S, H, Hkv, d_qk=d_qk, d_v=128, layout=layout,
                           seed=2000 + S + 7 * d_qk + (dt == "fp8"))
    t = workloads.make_inputs(w)
    O, L = run_gpu(t, w)
    Oref, Lref = run_oracle(t, w)
    assert_parity(O, L, Oref, Lref, dt, f"{dt} d{d_qk} {layout} B{B} S{S} H{H}/{Hkv}")
    _check_status()


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_activation_like_d192(dt):
    w = W[f"{dt}_mla_b1_h16_s16384_d192"].with_(S=1024, H=4, Hkv=4)
    t = workloads.make_inputs(w)
    O, L = run_gpu(t, w)
    Oref, Lref = run_oracle(t, w)
    assert_parity(O, L, Oref, Lref, dt, f"activation-like {dt} d192")


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_activation_like_d128_gqa(dt):
    # Peaked rows whose maximum keeps moving (outlier channels shared by q
    # and k): most tiles take the rescale path, whose P, sums and FP8 lo term
    # are recomputed in one pass; GQA 4:1, ragged length, bshd.
    w = workloads.Workload("activation_d128", dt, 1, 1500, 8, 2, layout="bshd",
                           values="activation", seed=3100 + (dt == "fp8"))
    t = workloads.make_inputs(w)
    O, L = run_gpu(t, w)
    Oref, Lref = run_oracle(t, w)
    assert_parity(O, L, Oref, Lref, dt, f"activation-like {dt} d128 GQA")
    O2, L2 = run_gpu(t, w)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    _check_status()


def test_explicit_scale():
    w = W["bf16_mha_b1_h2_s256_d128"].with_(S=300)
    t = workloads.make_inputs(w)
    O, L = run_gpu(t, w, scale=0.37)
    Oref, Lref = run_oracle(t, w, scale=0.37)
    assert_parity(O, L, Oref, Lref, "bf16", "scale 0.37")


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_deterministic(dt):
    w = W[f"{dt}_mha_b2_h32_s2048_d128"].with_(H=8, Hkv=2, S=1536)
    t = workloads.make_inputs(w)
    ref = run_gpu(t, w)
    for _ in range(4):
        O, L = run_gpu(t, w)
        assert np.array_equal(O, ref[0]) and np.array_equal(L, ref[1])


def test_serialized_pv_is_bitwise_equal():
    w = W["bf16_gqa_b1_h32kv8_s8192_d128"].with_(S=2048, H=8, Hkv=2)
    t = workloads.make_inputs(w)
    O1, L1 = run_gpu(t, w)
    assert zf.zyfa_set_option(zf.ZYFA_OPT_SERIALIZE_PV, 1) == 0
    try:
        O2, L2 = run_gpu(t, w)
    finally:
        zf.zyfa_set_option(zf.ZYFA_OPT_SERIALIZE_PV, 0)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_layouts_bitwise_equal():
    w = W["bf16_mha_b1_h2_s256_d128"].with_(S=700, H=4, Hkv=2, B=2)
    t = workloads.make_inputs(w)
    O1, L1 = run_gpu(t, w)
    t2 = {n: (t[n].transpose(1, 2).contiguous() if n in "qkv" else t[n]) for n in t}
    O2, L2 = run_gpu(t2, w.with_(layout="bhsd"))
    assert np.array_equal(to_bhsd(O1, "bshd"), O2) and np.array_equal(L1, L2)


def test_gqa_equals_repeated_mha_bitwise():
    w = W["bf16_gqa_b1_h32kv8_s8192_d128"].with_(S=600, H=8, Hkv=2)
    t = workloads.make_inputs(w)
    O1, L1 = run_gpu(t, w)
    rep = {n: (t[n].repeat_interleave(4, dim=2) if n in "kv" else t[n]) for n in t}
    O2, L2 = run_gpu(rep, w.with_(Hkv=8))
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_ragged_equals_zero_padded_bitwise():
    w = W["bf16_mha_b1_h2_s256_d128"].with_(S=1000, H=2, Hkv=2)
    t = workloads.make_inputs(w)
    O1, L1 = run_gpu(t, w)
    pad = 1024 - 1000
    tp = {n: (torch.cat([t[n], torch.zeros_like(t[n][:, :pad])], dim=1) if n in "qkv" else t[n])
          for n in t}
    O2, L2 = run_gpu(tp, w.with_(S=1024))
    assert np.array_equal(O1, O2[:, :1000]) and np.array_equal(L1, L2[:, :, :1000])


def test_descales_read_from_device_memory():
    """Changing the device descale values changes the result with no new host values."""
    w = W["fp8_gqa_b1_h32kv8_s16384_d128"].with_(S=512, H=4, Hkv=2)
    t = workloads.make_inputs(w)
    from gpu_util import device_inputs
    q, k, v, ds = device_inputs(t, w)
    out1, lse1 = zf.attention(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2],
                              return_lse=True)
    ds[2].mul_(2.0)           # v_descale doubled on the device
    out2, lse2 = zf.attention(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2],
                              return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(lse1, lse2)
    assert torch.allclose(out2.float(), 2 * out1.float(), rtol=0, atol=0)
