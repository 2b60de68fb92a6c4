"""Single-feature probes of the tensor-core encodings (TMA 128-byte swizzle,
shared-memory and instruction descriptors, A operand in tensor memory, V as
an MN-major operand), each against a float64 CPU product."""

import ctypes
import os

import numpy as np
import pytest
import torch

from causal_flashattention_prefill_gb300 import build as zbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def probes():
    path = zbuild.build_probes()
    lib = ctypes.CDLL(path)
    lib.zyfa_probe_mma.restype = ctypes.c_int
    lib.zyfa_probe_mma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def _operands(f8: bool, seed: int):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(128, 128, generator=g)
    b = torch.randn(128, 128, generator=g)
    if f8:
        a, b = (x.mul(8.0).to(torch.float8_e4m3fn) for x in (a, b))
    else:
        a, b = (x.to(torch.bfloat16) for x in (a, b))
    return a, b


@pytest.mark.parametrize("f8", [0, 1], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("mode", [0, 1], ids=["ss_kmajor", "ts_mnmajor"])
def test_probe_mma(probes, f8, mode):
    a, b = _operands(bool(f8), 7 + 2 * f8 + mode)
    da, db = a.cuda(), b.cuda()
    d = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = probes.zyfa_probe_mma(f8, mode, da.data_ptr(), db.data_ptr(), d.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    A = a.to(torch.float64).numpy()
    B = b.to(torch.float64).numpy()
    ref = A @ B.T if mode == 0 else A @ B
    got = d.cpu().double().numpy()
    err = np.abs(got - ref)
    print(f"f8={f8} mode={mode} max|err|={err.max():.3e} max|ref|={np.abs(ref).max():.3e}")
    assert np.all(np.isfinite(got))
    # FP32 accumulation of 128 exact products
    assert err.max() <= 1e-5 * np.abs(ref).max() * 128 ** 0.5 + 1e-6


def test_bounded_wait_runs_out_and_reports(probes):
    """Failure detection without a GPU fault: a wait whose arrival never comes
    ends after its limit with an error status the host reads, the abort flag
    raised for the other roles, and the context still usable."""
    probes.zyfa_probe_wait_timeout.restype = ctypes.c_int
    probes.zyfa_probe_wait_timeout.argtypes = [ctypes.c_void_p]
    probes.zyfa_probe_status.restype = ctypes.c_int
    probes.zyfa_probe_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
    probes.zyfa_probe_status_reset.restype = ctypes.c_int
    assert probes.zyfa_probe_status_reset() == 0
    out = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    assert probes.zyfa_probe_wait_timeout(out.data_ptr()) == 0
    ok, aborted, us = out.cpu().tolist()
    assert ok == 0 and aborted == 1
    assert 1_000_000 <= us <= 10_000_000      # the 2 s limit, measured on the GPU clock
    v = ctypes.c_int(0)
    assert probes.zyfa_probe_status(ctypes.byref(v)) == 0 and v.value & 1
    assert probes.zyfa_probe_status_reset() == 0
    # the context is still usable: a small attention call succeeds
    import causal_flashattention_prefill_gb300 as zf
    q = torch.randn(1, 300, 2, 128, device="cuda").to(torch.bfloat16)
    o = zf.flash_attn_func(q, q, q)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
