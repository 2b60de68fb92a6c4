"""Torch-level wrappers over the C ABI.

PyTorch supplies device memory and the current stream; the attention runs in
the CUDA library only.  ``flash_attn_func`` follows the calling conventions
the ZYFA README lists ("Usage", "Differences from flash-attn").
"""

from __future__ import annotations

import math

import torch

from . import _lib


class ZyfaError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, status: int):
        super().__init__(f"zyfa status {status}: {_lib.zyfa_status_string(status)}")
        self.status = status


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.ZYFA_BF16
    if t.dtype == torch.float8_e4m3fn:
        return _lib.ZYFA_FP8_E4M3
    raise TypeError(f"unsupported input dtype {t.dtype}: BF16 or float8_e4m3fn only")


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def attention(q, k, v, out=None, lse=None, q_descale=None, k_descale=None, v_descale=None,
              softmax_scale=None, layout="bshd", return_lse=False, stream=None):
    """Causal forward attention on device tensors through ``zyfa_fwd_scaled``.

    ``q`` (B,S,H,d_qk) and ``k``/``v`` (B,S,Hkv,d) for ``layout="bshd"``, or
    (B,H,S,d) for ``"bhsd"``; BF16 or float8_e4m3fn, contiguous.  FP8 needs
    three 1-element float32 device descale tensors.  ``out``/``lse`` are
    allocated when not given.  Returns ``out`` or ``(out, lse)``.
    """
    dt = _dtype_code(q)
    if not (k.dtype == q.dtype and v.dtype == q.dtype):
        raise TypeError("q, k and v must have the same dtype")
    lay = {"bshd": _lib.ZYFA_BSHD, "bhsd": _lib.ZYFA_BHSD}[layout]
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    if lay == _lib.ZYFA_BSHD:
        B, S, H, d_qk = q.shape
        Hkv, d_v = k.shape[2], v.shape[3]
        out_shape = (B, S, H, d_v)
    else:
        B, H, S, d_qk = q.shape
        Hkv, d_v = k.shape[1], v.shape[3]
        out_shape = (B, H, S, d_v)
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    if out is None:
        out = torch.empty(out_shape, dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d_qk)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    st = _lib.zyfa_fwd_scaled(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, Hkv,
                              d_qk, d_v, dt, _ptr(q_descale), _ptr(k_descale), _ptr(v_descale),
                              float(softmax_scale), lay, stream)
    if st != _lib.ZYFA_OK:
        raise ZyfaError(st)
    return (out, lse) if return_lse else out


def fp8_quantize(x: torch.Tensor, workspace: torch.Tensor = None, stream=None):
    """Per-tensor e4m3 quantisation with a power-of-two descale, on the GPU.

    Returns ``(x8, descale)``: ``x8`` a ``float8_e4m3fn`` tensor shaped like
    ``x`` and ``descale`` a 1-element float32 tensor on ``x``'s device,
    ``2**ceil(log2(max|x| / 448))``; the call never waits for the host
    (ZYFA README, "Usage").  ``x`` is BF16 or float32, contiguous.
    """
    if x.dtype == torch.bfloat16:
        xt = _lib.ZYFA_BF16
    elif x.dtype == torch.float32:
        xt = _lib.ZYFA_F32
    else:
        raise TypeError(f"fp8_quantize takes BF16 or float32, not {x.dtype}")
    x = x.detach().contiguous()
    x8 = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    descale = torch.empty(1, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(_lib.zyfa_fp8_quantize_workspace_bytes(), dtype=torch.uint8,
                                device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    st = _lib.zyfa_fp8_quantize(x.data_ptr(), x.numel(), xt, x8.data_ptr(), descale.data_ptr(),
                                workspace.data_ptr(), stream)
    if st != _lib.ZYFA_OK:
        raise ZyfaError(st)
    return x8, descale


class _NoBackward(torch.autograd.Function):
    @staticmethod
    def forward(ctx, out, *inputs):
        return out

    @staticmethod
    def backward(ctx, *grads):
        raise RuntimeError("causal prefill attention has no backward pass")


def _descale_tensor(d, device):
    if d is None:
        return None
    if isinstance(d, (int, float)):
        return torch.full((1,), float(d), dtype=torch.float32, device=device)
    if not isinstance(d, torch.Tensor) or d.dtype != torch.float32:
        raise TypeError("a descale is a Python float or a float32 tensor")
    # A (B, Hkv) expansion of one value is read through its first element.
    return d.reshape(-1)[:1] if d.numel() > 1 else d.reshape(1)


def flash_attn_func(q, k, v, dropout_p=0.0, softmax_scale=None, causal=True,
                    window_size=(-1, -1), q_descale=None, k_descale=None, v_descale=None,
                    layout="bshd", return_lse=False, return_attn_probs=False):
    """flash-attn 2 argument order; causal only; BF16 or FP8 inputs, BF16 out."""
    if isinstance(softmax_scale, bool) or not isinstance(dropout_p, (int, float)):
        raise TypeError("arguments follow flash-attn 2's order (q, k, v, dropout_p, "
                        "softmax_scale, causal, ...); pass the others by keyword")
    if dropout_p != 0.0:
        raise ValueError("dropout is not supported")
    if causal is not True:
        raise ValueError("only causal attention is supported: pass causal=True")
    if tuple(window_size) not in ((-1, -1), (-1, 0), (None, None)):
        raise ValueError("sliding windows are not supported")
    fp8 = q.dtype == torch.float8_e4m3fn
    if fp8 and (q_descale is None or k_descale is None or v_descale is None):
        raise ValueError("FP8 inputs need q_descale, k_descale and v_descale")
    q, k, v = (t.contiguous() for t in (q, k, v))
    dq, dk, dv = (_descale_tensor(d, q.device) for d in (q_descale, k_descale, v_descale))
    want_lse = return_lse or return_attn_probs
    res = attention(q, k, v, q_descale=dq, k_descale=dk, v_descale=dv,
                    softmax_scale=softmax_scale, layout=layout, return_lse=want_lse)
    out, lse = res if want_lse else (res, None)
    if torch.is_grad_enabled() and any(t.requires_grad for t in (q, k, v)):
        out = _NoBackward.apply(out, q, k, v)
    if return_attn_probs:
        return out, lse, None
    if return_lse:
        return out, lse
    return out
