"""The seeded input generators: reproducibility and the FP8 quantisation rule."""

import math

import numpy as np
import torch

import workloads


def test_seeds_reproducible():
    w = workloads.WORKLOADS["bf16_mha_b1_h2_s256_d128"]
    a, b = workloads.make_inputs(w), workloads.make_inputs(w)
    for n in ("q", "k", "v"):
        assert torch.equal(a[n], b[n])
    assert not torch.equal(a["q"], a["k"])


def test_shapes_follow_layout():
    w = workloads.WORKLOADS["bf16_mla_b1_h16_s16384_d192"].with_(S=40, H=4, Hkv=2)
    t = workloads.make_inputs(w)
    assert t["q"].shape == (1, 4, 40, 192)
    assert t["k"].shape == (1, 2, 40, 192)
    assert t["v"].shape == (1, 2, 40, 128)
    w2 = workloads.WORKLOADS["bf16_gqa_b1_h32kv8_s8192_d128"].with_(S=40)
    t2 = workloads.make_inputs(w2)
    assert t2["q"].shape == (1, 40, 32, 128) and t2["k"].shape == (1, 40, 8, 128)


def test_fp8_descale_power_of_two_and_tight():
    for seed in range(5):
        x = workloads.gaussian((3, 77, 5), 50 + seed) * (seed + 0.3)
        codes, ds = workloads.fp8_quantize_cpu(x)
        e = math.log2(ds)
        assert e == int(e)
        amax = float(x.abs().max())
        assert 224.0 < amax / ds <= 448.0
        deq = codes.to(torch.float64) * ds
        assert torch.all(torch.isfinite(deq))
        # round to nearest: error at most half a step of e4m3 (3 mantissa bits)
        err = (deq - x.double()).abs()
        assert torch.all(err <= torch.maximum(x.double().abs() * 2 ** -4, torch.tensor(2.0 ** -10 * ds)))


def test_activation_like_has_outliers():
    w = workloads.WORKLOADS["bf16_mla_b1_h16_s16384_d192"].with_(S=256)
    q, k, _ = workloads.fp32_inputs(w)
    sq = q.float().pow(2).mean(dim=(0, 1, 2)).sqrt()
    sk = k.float().pow(2).mean(dim=(0, 1, 2)).sqrt()
    top_q = set(torch.topk(sq, 4).indices.tolist())
    top_k = set(torch.topk(sk, 4).indices.tolist())
    assert top_q == top_k          # outlier channels shared by q and k
    assert float(sq.max()) > 10.0


def test_sample_rows_cover_edges():
    rows = workloads.sample_rows(1000, 1)
    assert rows[0] == 0 and rows[-1] == 999
    for r in (127, 128, 129, 255, 256, 257, 895, 896, 897):
        assert r in rows
    assert np.all(np.diff(rows) > 0)


def test_flops_formula():
    w = workloads.WORKLOADS["bf16_gqa_b1_h32kv8_s16384_d128"]
    assert w.flops == 1 * 32 * 16384 ** 2 * 256
