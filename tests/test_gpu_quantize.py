"""The GPU FP8 quantiser (zyfa_fp8_quantize) against the oracle's encoder:
e4m3 bytes and descale bit-exact, for BF16 and FP32 inputs."""

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads
from oracle.formats import bf16_to_f64
from oracle.quantize import fp8_quantize_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()


def _check(x_host: torch.Tensor):
    x8, ds = zf.fp8_quantize(x_host.cuda())
    torch.cuda.synchronize()
    got = x8.view(torch.uint8).cpu().numpy().reshape(-1)
    if x_host.dtype == torch.bfloat16:
        xf = bf16_to_f64(x_host.view(torch.int16).numpy().view(np.uint16)).reshape(-1)
    else:
        xf = x_host.double().numpy().reshape(-1)
    ref, dref = fp8_quantize_f64(xf)
    assert float(ds.item()) == dref
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} codes differ"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [1, 7, 8, 9, 255, 1000, 4097, (1 << 20) + 3])
def test_quantize_random(dtype, n):
    x = workloads.gaussian((n,), 500 + n) * 3.0
    _check(x.to(dtype))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_large_tensor(dtype):
    x = workloads.gaussian((16, 1024, 1024), 77)
    _check(x.to(dtype))


def test_quantize_boundaries():
    # amax exactly 448 * 2^k, just above it, ties between e4m3 values, -0.0
    for amax in (448.0, 448.0 * 4, 449.0, 224.0, 1.0, 2.0 ** -20):
        x = torch.tensor([0.0, -0.0, amax, -amax / 3, amax / 7, 1.0625 * amax / 448,
                          1.1875 * amax / 448], dtype=torch.float32)
        _check(x)
    _check(torch.zeros(1000, dtype=torch.float32))


def test_quantize_deterministic():
    x = (workloads.gaussian((1 << 22,), 9) * 11.0).to(torch.bfloat16).cuda()
    a, da = zf.fp8_quantize(x)
    for _ in range(3):
        b, db = zf.fp8_quantize(x)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)) and torch.equal(da, db)
