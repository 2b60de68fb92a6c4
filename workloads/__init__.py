"""Seeded synthetic inputs shared by the tests, ``smoke()`` and ``bench.py``.

This module only draws numbers and stores them in the input formats (BF16, or
e4m3 with one power-of-two descale per tensor).  It contains none of the
attention arithmetic, so the oracle and the CUDA path can both consume its
output without sharing any computation.

Shapes, value distributions and seeds:

* Gaussian workloads: q, k, v i.i.d. N(0, 1) in FP32, then rounded to BF16
  (round to nearest even) or quantised to e4m3.
* Activation-like workloads (the MLA-form case with d_qk = 192): q and k are
  N(0, 1) times a per-channel factor drawn from LogNormal(0, 0.5) once per
  tensor, and 4 outlier channels (indices drawn once, shared by q and k) are
  multiplied by 20; v is N(0, 1).  They stand in for the captured post-RoPE
  activations that the ZYFA README times ("Captured activations at sustained
  clocks"), which are not available here.
* FP8 quantisation uses one power-of-two descale per tensor,
  ``descale = 2**ceil(log2(max|x| / 448))``, so ``max|x| / descale <= 448``
  (448 is the largest finite e4m3 value), and rounds ``x / descale`` to the
  nearest e4m3 value (ties to even).

All draws use ``torch.Generator().manual_seed(seed)`` on the CPU, so the bytes
are identical on every machine.  ``seed = base + tensor_index`` with
q = 0, k = 1, v = 2 and the outlier-channel draw = 3.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    """One synthetic attention problem (sizes, formats and value recipe)."""

    name: str
    dtype: str            # "bf16" or "fp8"
    B: int
    S: int
    H: int
    Hkv: int
    d_qk: int = 128
    d_v: int = 128
    layout: str = "bshd"  # "bshd" or "bhsd"
    values: str = "gaussian"   # "gaussian" or "activation"
    seed: int = 1000

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def flops(self) -> float:
        """Causal forward FLOPs, 2*B*H*(S^2/2)*(d_qk+d_v)."""
        return 2.0 * self.B * self.H * (self.S * self.S / 2.0) * (self.d_qk + self.d_v)


def _named() -> dict:
    w = {}
    w["bf16_mha_b1_h2_s256_d128"] = Workload(
        "bf16_mha_b1_h2_s256_d128", "bf16", 1, 256, 2, 2, seed=1010)
    w["bf16_gqa_b1_h32kv8_s8192_d128"] = Workload(
        "bf16_gqa_b1_h32kv8_s8192_d128", "bf16", 1, 8192, 32, 8, seed=1020)
    w["fp8_gqa_b1_h32kv8_s16384_d128"] = Workload(
        "fp8_gqa_b1_h32kv8_s16384_d128", "fp8", 1, 16384, 32, 8, seed=1030)
    w["bf16_gqa_b1_h32kv8_s16384_d128"] = Workload(
        "bf16_gqa_b1_h32kv8_s16384_d128", "bf16", 1, 16384, 32, 8, seed=1035)
    for dt in ("bf16", "fp8"):
        n = f"{dt}_mla_b1_h16_s16384_d192"
        w[n] = Workload(n, dt, 1, 16384, 16, 16, d_qk=192, d_v=128,
                        layout="bhsd", values="activation", seed=1040)
        for S in (2048, 4096, 16384, 30000, 32768):
            n = f"{dt}_mha_b2_h32_s{S}_d128"
            w[n] = Workload(n, dt, 2, S, 32, 32, seed=1050 + (S % 97))
    return w


WORKLOADS = _named()


def gaussian(shape, seed: int) -> torch.Tensor:
    """FP32 N(0, 1) draws from a fresh CPU generator."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def fp8_quantize_cpu(x: torch.Tensor):
    """Per-tensor power-of-two e4m3 quantisation: returns (codes, descale).

    ``codes`` is a ``torch.float8_e4m3fn`` tensor, ``descale`` a Python float
    with ``x ~= codes * descale``.
    """
    amax = float(x.abs().max())
    if amax == 0.0:
        descale = 1.0
    else:
        descale = 2.0 ** math.ceil(math.log2(amax / E4M3_MAX))
    codes = (x / descale).to(torch.float8_e4m3fn)
    return codes, descale


def _shapes(w: Workload):
    if w.layout == "bshd":
        return ((w.B, w.S, w.H, w.d_qk), (w.B, w.S, w.Hkv, w.d_qk),
                (w.B, w.S, w.Hkv, w.d_v))
    return ((w.B, w.H, w.S, w.d_qk), (w.B, w.Hkv, w.S, w.d_qk),
            (w.B, w.Hkv, w.S, w.d_v))


def _activation_like(shape, seed: int, outliers: torch.Tensor) -> torch.Tensor:
    d = shape[-1]
    x = gaussian(shape, seed)
    g = torch.Generator().manual_seed(int(seed) + 100)
    f = torch.exp(0.5 * torch.randn(d, generator=g, dtype=torch.float32))
    f[outliers] *= 20.0
    return x * f


def fp32_inputs(w: Workload):
    """The FP32 draws (q, k, v) before rounding to the input format."""
    sq, sk, sv = _shapes(w)
    if w.values == "gaussian":
        return gaussian(sq, w.seed + 0), gaussian(sk, w.seed + 1), gaussian(sv, w.seed + 2)
    if w.values == "activation":
        g = torch.Generator().manual_seed(w.seed + 3)
        outliers = torch.randperm(w.d_qk, generator=g)[:4]
        return (_activation_like(sq, w.seed + 0, outliers),
                _activation_like(sk, w.seed + 1, outliers),
                gaussian(sv, w.seed + 2))
    raise ValueError(f"unknown value recipe {w.values!r}")


def make_inputs(w: Workload) -> dict:
    """Host tensors for ``w``: q, k, v in the input format, plus descales.

    BF16 workloads return ``torch.bfloat16`` tensors and descales of 1.0;
    FP8 workloads return ``torch.float8_e4m3fn`` tensors and the three
    power-of-two descales.
    """
    q, k, v = fp32_inputs(w)
    if w.dtype == "bf16":
        return dict(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16),
                    v=v.to(torch.bfloat16), q_descale=1.0, k_descale=1.0,
                    v_descale=1.0)
    if w.dtype == "fp8":
        (q8, qs), (k8, ks), (v8, vs) = (fp8_quantize_cpu(t) for t in (q, k, v))
        return dict(q=q8, k=k8, v=v8, q_descale=qs, k_descale=ks, v_descale=vs)
    raise ValueError(f"unknown dtype {w.dtype!r}")


def codes(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a BF16 (uint16) or e4m3 (uint8) tensor, as numpy."""
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.contiguous().view(torch.uint8).numpy()
    raise TypeError(f"no code view for {t.dtype}")


def sample_rows(S: int, seed: int, n_random: int = 512) -> np.ndarray:
    """Query rows to check on large problems.

    Rows 0..255, every 128-row tile boundary +-1, the last 256 rows and
    ``n_random`` seeded random rows, sorted and de-duplicated.
    """
    rows = set(range(min(S, 256)))
    for t in range(0, S + 1, 128):
        for r in (t - 1, t, t + 1):
            if 0 <= r < S:
                rows.add(r)
    rows.update(range(max(0, S - 256), S))
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, S, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)
