"""The default-scale entry point ``zyfa_fwd`` called directly through the C
ABI (ctypes, device pointers), for both input formats and both head-dim
forms, against the float64 oracle at its default scale 1/sqrt(d_qk) (the
flash-attn convention the ZYFA README follows in "Usage"; the pages print no
other default).  ``zyfa_fwd_scaled`` with that scale written out must give
the same bits."""

import math

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads
from gpu_util import assert_parity, device_inputs, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()


def _call(fn, w, q, k, v, ds, out, lse, *scale):
    lay = zf.ZYFA_BSHD if w.layout == "bshd" else zf.ZYFA_BHSD
    dt = zf.ZYFA_BF16 if w.dtype == "bf16" else zf.ZYFA_FP8_E4M3
    p = [0 if d is None else d.data_ptr() for d in ds]
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), w.B, w.S,
            w.H, w.Hkv, w.d_qk, w.d_v, dt, p[0], p[1], p[2], *scale, lay,
            torch.cuda.current_stream().cuda_stream)
    assert st == zf.ZYFA_OK, zf.zyfa_status_string(st)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("d_qk,layout", [(128, "bshd"), (192, "bhsd")])
def test_zyfa_fwd_default_scale(dtype, d_qk, layout):
    w = workloads.Workload("entry", dtype, 2, 777, 4, 2, d_qk=d_qk, d_v=128, layout=layout,
                           seed=4100 + d_qk + (dtype == "fp8"))
    t = workloads.make_inputs(w)
    q, k, v, ds = device_inputs(t, w)
    oshape = (w.B, w.S, w.H, w.d_v) if layout == "bshd" else (w.B, w.H, w.S, w.d_v)
    out = torch.empty(oshape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=q.device)
    _call(zf.zyfa_fwd, w, q, k, v, ds, out, lse)
    torch.cuda.synchronize()
    O = out.float().cpu().double().numpy()
    L = lse.cpu().double().numpy()
    Oref, Lref = run_oracle(t, w)        # the oracle's own default scale
    assert_parity(O, L, Oref, Lref, dtype, f"zyfa_fwd {dtype} d{d_qk} {layout}")
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    _call(zf.zyfa_fwd_scaled, w, q, k, v, ds, out2, lse2, 1.0 / math.sqrt(d_qk))
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
