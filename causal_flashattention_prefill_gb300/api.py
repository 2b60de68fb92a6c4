"""Torch-level wrappers over the C ABI.

PyTorch supplies device memory and the current stream; the attention runs in
the CUDA library only.  ``flash_attn_func`` and its packed and varlen forms
follow the calling conventions the ZYFA README lists ("Usage", "Differences
from flash-attn") and reach the library through the custom operator
``torch.ops.zyfa.fwd``.
"""

from __future__ import annotations

from typing import Optional, Tuple

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
    """Causal forward attention on device tensors through the C ABI.

    ``q`` (B,S,H,d_qk) and ``k``/``v`` (B,S,Hkv,d) for ``layout="bshd"``, or
    (B,H,S,d) for ``"bhsd"``; BF16 or float8_e4m3fn, contiguous.  FP8 needs
    three 1-element float32 device descale tensors.  ``out``/``lse`` are
    allocated when not given.  Without ``softmax_scale`` the call goes to
    ``zyfa_fwd``, which applies the default scale itself; with one, to
    ``zyfa_fwd_scaled``.  Returns ``out`` or ``(out, lse)``.
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
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, Hkv, d_qk, d_v, dt,
            _ptr(q_descale), _ptr(k_descale), _ptr(v_descale))
    if softmax_scale is None:
        st = _lib.zyfa_fwd(*args, lay, stream)
    else:
        st = _lib.zyfa_fwd_scaled(*args, float(softmax_scale), lay, stream)
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


def _descale_tensor(d, device):
    if d is None:
        return None
    if isinstance(d, (int, float)):
        return torch.full((1,), float(d), dtype=torch.float32, device=device)
    if not isinstance(d, torch.Tensor) or d.dtype != torch.float32:
        raise TypeError("a descale is a Python float or a float32 tensor")
    # A (B, Hkv) expansion of one value is read through its first element.
    return d.reshape(-1)[:1] if d.numel() > 1 else d.reshape(1)


# The attention is registered as the custom operator torch.ops.zyfa.fwd (ZYFA
# README, "Usage"), so torch.compile traces through calls and they can be
# captured in CUDA graphs (the library allocates nothing and never waits for
# the host).  The fake implementation gives torch.compile the output shapes.
# The LSE output is a (0,)-shaped tensor when it is not requested.
@torch.library.custom_op("zyfa::fwd", mutates_args=())
def _fwd_op(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
            q_descale: Optional[torch.Tensor], k_descale: Optional[torch.Tensor],
            v_descale: Optional[torch.Tensor], softmax_scale: Optional[float], layout: str,
            return_lse: bool) -> Tuple[torch.Tensor, torch.Tensor]:
    res = attention(q, k, v, q_descale=q_descale, k_descale=k_descale, v_descale=v_descale,
                    softmax_scale=softmax_scale, layout=layout, return_lse=return_lse)
    if return_lse:
        return res
    return res, torch.empty(0, dtype=torch.float32, device=q.device)


def _out_lse_shapes(q, v, layout):
    if layout == "bshd":
        B, S, H, _ = q.shape
        return (B, S, H, v.shape[3]), (B, H, S)
    B, H, S, _ = q.shape
    return (B, H, S, v.shape[3]), (B, H, S)


@_fwd_op.register_fake
def _(q, k, v, q_descale, k_descale, v_descale, softmax_scale, layout, return_lse):
    o_shape, l_shape = _out_lse_shapes(q, v, layout)
    out = q.new_empty(o_shape, dtype=torch.bfloat16)
    lse = q.new_empty(l_shape if return_lse else (0,), dtype=torch.float32)
    return out, lse


def _fwd_backward(ctx, *grads):
    raise RuntimeError("causal prefill attention has no backward pass")


_fwd_op.register_autograd(_fwd_backward)


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
    if layout not in ("bshd", "bhsd"):
        raise ValueError(f"layout is 'bshd' or 'bhsd', not {layout!r}")
    q, k, v = (t.contiguous() for t in (q, k, v))
    dq, dk, dv = (_descale_tensor(d, q.device) for d in (q_descale, k_descale, v_descale))
    if softmax_scale is not None:
        softmax_scale = float(softmax_scale)
    want_lse = bool(return_lse or return_attn_probs)
    out, lse = torch.ops.zyfa.fwd(q, k, v, dq, dk, dv, softmax_scale, layout, want_lse)
    if not want_lse:
        lse = None
    if return_attn_probs:
        return out, lse, None
    if return_lse:
        return out, lse
    return out


def _check_unsupported(softcap=0.0, alibi_slopes=None, deterministic=False, block_table=None):
    if softcap not in (0, 0.0, None):
        raise ValueError("softcap is not supported")
    if alibi_slopes is not None:
        raise ValueError("ALiBi is not supported")
    if block_table is not None:
        raise ValueError("paged KV is not supported")
    # Every result is deterministic, so `deterministic` needs no action.


def flash_attn_qkvpacked_func(qkv, dropout_p=0.0, softmax_scale=None, causal=True,
                              window_size=(-1, -1), softcap=0.0, alibi_slopes=None,
                              deterministic=False, return_attn_probs=False, q_descale=None,
                              k_descale=None, v_descale=None, return_lse=False):
    """flash-attn's packed form: ``qkv`` is (batch, seqlen, 3, nheads, headdim)
    (MHA, d_qk = d_v).  The three slices are copied to contiguous tensors
    before the kernel runs (ZYFA README, "Differences from flash-attn")."""
    _check_unsupported(softcap, alibi_slopes, deterministic)
    if qkv.dim() != 5 or qkv.shape[2] != 3:
        raise ValueError("qkv must be (batch, seqlen, 3, nheads, headdim)")
    q, k, v = qkv.unbind(dim=2)
    return flash_attn_func(q, k, v, dropout_p, softmax_scale, causal, window_size,
                           q_descale=q_descale, k_descale=k_descale, v_descale=v_descale,
                           return_lse=return_lse, return_attn_probs=return_attn_probs)


def flash_attn_kvpacked_func(q, kv, dropout_p=0.0, softmax_scale=None, causal=True,
                             window_size=(-1, -1), softcap=0.0, alibi_slopes=None,
                             deterministic=False, return_attn_probs=False, q_descale=None,
                             k_descale=None, v_descale=None, return_lse=False):
    """flash-attn's packed-KV form: ``q`` (batch, seqlen, nheads, headdim),
    ``kv`` (batch, seqlen, 2, nheads_k, headdim) (d_qk = d_v)."""
    _check_unsupported(softcap, alibi_slopes, deterministic)
    if kv.dim() != 5 or kv.shape[2] != 2:
        raise ValueError("kv must be (batch, seqlen, 2, nheads_k, headdim)")
    k, v = kv.unbind(dim=2)
    return flash_attn_func(q, k, v, dropout_p, softmax_scale, causal, window_size,
                           q_descale=q_descale, k_descale=k_descale, v_descale=v_descale,
                           return_lse=return_lse, return_attn_probs=return_attn_probs)


def _equal_segments(cu_seqlens, max_seqlen, total, name):
    """Batch size of an equal-length varlen batch; checks the metadata that can
    be checked without waiting for the device."""
    if max_seqlen <= 0 or total % max_seqlen != 0:
        raise ValueError(f"{name}: sequences must all have length max_seqlen "
                         f"({total} tokens, max_seqlen {max_seqlen})")
    batch = total // max_seqlen
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() != batch + 1:
        raise ValueError(f"{name}: cu_seqlens must hold batch + 1 = {batch + 1} offsets")
    if cu_seqlens.device.type == "cpu":
        want = torch.arange(0, total + 1, max_seqlen, dtype=cu_seqlens.dtype)
        if not torch.equal(cu_seqlens, want):
            raise ValueError(f"{name}: only sequences of equal length are supported")
    return batch


def flash_attn_varlen_func(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           dropout_p=0.0, softmax_scale=None, causal=True, window_size=(-1, -1),
                           softcap=0.0, alibi_slopes=None, deterministic=False,
                           return_attn_probs=False, block_table=None, q_descale=None,
                           k_descale=None, v_descale=None, return_lse=False):
    """flash-attn's varlen form for batches of equal-length sequences (ZYFA
    README, "Usage"): ``q`` (total, nheads, headdim), ``k``/``v`` (total,
    nheads_k, headdim), ``cu_seqlens_*`` = [0, S, 2S, ...].  Device-resident
    offsets are trusted (checking them would wait for the device); offsets on
    the host are checked.  Returns ``out`` (total, nheads, d_v) and, on
    request, the LSE as (nheads, total)."""
    _check_unsupported(softcap, alibi_slopes, deterministic, block_table)
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("varlen q, k, v are (total_tokens, heads, headdim)")
    if max_seqlen_q != max_seqlen_k or q.shape[0] != k.shape[0] or k.shape[0] != v.shape[0]:
        raise ValueError("causal prefill needs seqlen_q = seqlen_k for every sequence")
    batch = _equal_segments(cu_seqlens_q, max_seqlen_q, q.shape[0], "cu_seqlens_q")
    _equal_segments(cu_seqlens_k, max_seqlen_k, k.shape[0], "cu_seqlens_k")
    S = max_seqlen_q
    q4, k4, v4 = (t.reshape(batch, S, t.shape[1], t.shape[2]) for t in (q, k, v))
    want_lse = return_lse or return_attn_probs
    res = flash_attn_func(q4, k4, v4, dropout_p, softmax_scale, causal, window_size,
                          q_descale=q_descale, k_descale=k_descale, v_descale=v_descale,
                          return_lse=want_lse)
    out, lse = res if want_lse else (res, None)
    out = out.reshape(batch * S, out.shape[2], out.shape[3])
    if lse is not None:
        lse = lse.permute(1, 0, 2).reshape(lse.shape[1], batch * S)
    if return_attn_probs:
        return out, lse, None
    if return_lse:
        return out, lse
    return out


def hadamard_signs(d: int, seed: int = 0, device="cuda") -> torch.Tensor:
    """The random signs s of R = diag(s) H / sqrt(d), drawn as the ZYFA README
    draws them ("Using FP8 attention in a model": a seeded generator, one
    matrix for every layer and head), as a float32 tensor on ``device``."""
    g = torch.Generator().manual_seed(seed)
    s = torch.randint(0, 2, (d,), generator=g) * 2 - 1
    return s.to(dtype=torch.float32, device=device)


def fp8_quantize_rotated(x: torch.Tensor, signs: torch.Tensor, workspace: torch.Tensor = None,
                         stream=None):
    """Rotation then per-tensor e4m3 quantisation, on the GPU, for q and k.

    Each row of the last dimension d (128, or 192 in the DCT x Hadamard form)
    becomes ``x @ R`` with ``R = diag(signs) H / sqrt(d)``; the result is
    quantised like ``fp8_quantize``.  Rotate q and k with the same signs and
    leave v unrotated: the scores are unchanged and the quantisation error
    drops (ZYFA README, "Using FP8 attention in a model").  Returns
    ``(x8, descale)``.
    """
    if x.dtype == torch.bfloat16:
        xt = _lib.ZYFA_BF16
    elif x.dtype == torch.float32:
        xt = _lib.ZYFA_F32
    else:
        raise TypeError(f"fp8_quantize_rotated takes BF16 or float32, not {x.dtype}")
    d = x.shape[-1]
    if d not in (128, 192):
        raise ValueError(f"the rotation is defined for d = 128 and d = 192, not {d}")
    if signs.dtype != torch.float32 or signs.numel() != d or signs.device != x.device:
        raise ValueError("signs must be d float32 values on x's device")
    x = x.detach().contiguous()
    signs = signs.contiguous()
    x8 = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    descale = torch.empty(1, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(_lib.zyfa_fp8_quantize_workspace_bytes(), dtype=torch.uint8,
                                device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    st = _lib.zyfa_fp8_quantize_rotated(x.data_ptr(), x.numel() // d, d, xt, signs.data_ptr(),
                                        x8.data_ptr(), descale.data_ptr(), workspace.data_ptr(),
                                        stream)
    if st != _lib.ZYFA_OK:
        raise ZyfaError(st)
    return x8, descale
