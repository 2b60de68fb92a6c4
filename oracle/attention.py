"""Plain float64 causal attention that materialises the masked score matrix.

Test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference``) use it.

What it computes is the definition the ZYFA README states ("Usage" and
"Supported configurations"): causal forward attention with
``seqlen_q = seqlen_k``, i.e. for each batch ``b`` and query head ``h``

    Sc[i, j] = scale * <Q[b, h, i], K[b, hk, j]>      for j <= i
    Sc[i, j] = -inf                                    for j >  i
    P[i, :]  = exp(Sc[i, :] - m_i) / l_i,   m_i = max_j Sc[i, j],
                                            l_i = sum_j exp(Sc[i, j] - m_i)
    O[b, h, i] = sum_j P[i, j] * V[b, hk, j]
    LSE[b, h, i] = m_i + ln(l_i)   (natural-log log-sum-exp of the scaled
                                    scores, "return_lse" in "Usage")

with the grouped-query mapping ``hk = h // (H // Hkv)`` ("nheads a multiple of
nheads_k"; contiguous groups of query heads share one KV head, the flash-attn
convention that ZYFA's interface follows) and ``scale = 1/sqrt(d_qk)`` unless
given.  FP8 inputs enter as their exact dequantised values (e4m3 code value x
the tensor's descale).  The matrices are materialised in full (one ``S x S``
float64 matrix per (b, h)), with no tiling, online softmax or reordering.

Readings of points the pages leave open are listed with the design notes; the
ones used here: default scale ``1/sqrt(d_qk)``; key ``j`` is visible to query
``i`` iff ``j <= i`` (top-left equals bottom-right when the lengths are
equal); the LSE includes ``softmax_scale`` and the descales.

Pinned by ``tests/test_oracle.py``.
"""

from __future__ import annotations

import math

import numpy as np

from .formats import bf16_to_f64, e4m3_to_f64


def decode_inputs_f64(q, k, v, dtype: str = "bf16", layout: str = "bshd",
                      q_descale: float = 1.0, k_descale: float = 1.0,
                      v_descale: float = 1.0):
    """Exact float64 Q (B,H,S,dqk), K (B,Hkv,S,dqk), V (B,Hkv,S,dv).

    ``q``, ``k``, ``v`` are numpy arrays in the caller's layout: uint16 BF16
    bit patterns for ``dtype="bf16"``, uint8 e4m3 codes for ``dtype="fp8"``,
    or real numbers for ``dtype="f64"`` (taken as they are).
    """
    if dtype == "bf16":
        dq, dk, dv = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    elif dtype == "fp8":
        dq = e4m3_to_f64(q, q_descale)
        dk = e4m3_to_f64(k, k_descale)
        dv = e4m3_to_f64(v, v_descale)
    elif dtype == "f64":
        dq, dk, dv = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    if layout == "bshd":
        dq, dk, dv = (np.transpose(t, (0, 2, 1, 3)) for t in (dq, dk, dv))
    elif layout != "bhsd":
        raise ValueError(f"unknown layout {layout!r}")
    return (np.ascontiguousarray(dq), np.ascontiguousarray(dk),
            np.ascontiguousarray(dv))


def _kv_head(h: int, H: int, Hkv: int) -> int:
    if H % Hkv != 0:
        raise ValueError("H must be a multiple of Hkv")
    return h // (H // Hkv)


def causal_probs_f64(Qbh: np.ndarray, Kbh: np.ndarray, scale: float,
                     rows=None):
    """Masked scores, probabilities, row max and row sum for one (b, h).

    ``Qbh`` is (S, dqk), ``Kbh`` is (S, dqk).  ``rows`` selects query rows
    (default: all).  Returns ``(P, m, l)`` with ``P`` of shape
    (len(rows), S) holding the normalised probabilities (0 where masked).
    """
    S = Kbh.shape[0]
    rows = np.arange(Qbh.shape[0]) if rows is None else np.asarray(rows)
    sc = scale * (Qbh[rows] @ Kbh.T)                      # (r, S)
    visible = np.arange(S)[None, :] <= rows[:, None]      # j <= i
    sc = np.where(visible, sc, -np.inf)
    m = sc.max(axis=1)
    e = np.exp(sc - m[:, None])                           # exp(-inf) = 0
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def attention_rows_f64(q, k, v, rows=None, dtype: str = "bf16",
                       layout: str = "bshd", scale: float | None = None,
                       q_descale: float = 1.0, k_descale: float = 1.0,
                       v_descale: float = 1.0):
    """O and LSE for the selected query rows of every (b, h).

    Returns ``O`` of shape (B, H, R, dv) and ``LSE`` of shape (B, H, R),
    R = len(rows) (all rows when ``rows`` is None), in float64.
    """
    Q, K, V = decode_inputs_f64(q, k, v, dtype, layout,
                                q_descale, k_descale, v_descale)
    B, H, S, dqk = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(dqk)
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.empty((B, H, len(rows), dv), dtype=np.float64)
    LSE = np.empty((B, H, len(rows)), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            hk = _kv_head(h, H, Hkv)
            P, m, l = causal_probs_f64(Q[b, h], K[b, hk], scale, rows)
            O[b, h] = P @ V[b, hk]
            LSE[b, h] = m + np.log(l)
    return O, LSE


def attention_f64(q, k, v, dtype: str = "bf16", layout: str = "bshd",
                  scale: float | None = None, q_descale: float = 1.0,
                  k_descale: float = 1.0, v_descale: float = 1.0):
    """Full causal attention: ``O`` in the caller's layout and ``LSE`` (B,H,S).

    ``O`` is (B, S, H, dv) for ``layout="bshd"`` and (B, H, S, dv) for
    ``"bhsd"``, in float64.
    """
    O, LSE = attention_rows_f64(q, k, v, None, dtype, layout, scale,
                                q_descale, k_descale, v_descale)
    if layout == "bshd":
        O = np.ascontiguousarray(np.transpose(O, (0, 2, 1, 3)))
    return O, LSE
