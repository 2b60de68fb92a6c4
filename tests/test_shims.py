"""Host-side behaviour of the flash-attn style wrappers (no GPU): argument
checks that must fail before any launch, and the shapes the custom operator
reports to torch.compile (its fake implementation)."""

import pytest
import torch
from torch._subclasses.fake_tensor import FakeTensorMode

import causal_flashattention_prefill_gb300 as zf


def _bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def test_varlen_rejects_unequal_lengths_on_host():
    q = _bf16(30, 4, 128)
    cu = torch.tensor([0, 10, 30], dtype=torch.int32)
    with pytest.raises(ValueError, match="max_seqlen|equal length"):
        zf.flash_attn_varlen_func(q, q, q, cu, cu, 20, 20)
    cu = torch.tensor([0, 12, 24], dtype=torch.int32)  # right count, wrong offsets
    q = _bf16(24, 4, 128)
    with pytest.raises(ValueError, match="equal length"):
        zf.flash_attn_varlen_func(q, q, q, torch.tensor([0, 10, 24], dtype=torch.int32), cu, 12, 12)


def test_varlen_rejects_wrong_offset_count_and_cross_lengths():
    q = _bf16(24, 4, 128)
    with pytest.raises(ValueError, match="batch \\+ 1"):
        zf.flash_attn_varlen_func(q, q, q, torch.tensor([0, 24], dtype=torch.int32),
                                  torch.tensor([0, 24], dtype=torch.int32), 12, 12)
    cu = torch.tensor([0, 12, 24], dtype=torch.int32)
    with pytest.raises(ValueError, match="seqlen_q = seqlen_k"):
        zf.flash_attn_varlen_func(q, q, q, cu, cu, 12, 24)
    with pytest.raises(ValueError, match="total_tokens"):
        zf.flash_attn_varlen_func(_bf16(1, 24, 4, 128), q, q, cu, cu, 12, 12)


def test_packed_shapes_are_checked():
    with pytest.raises(ValueError, match="qkv must be"):
        zf.flash_attn_qkvpacked_func(_bf16(1, 8, 2, 4, 128))
    with pytest.raises(ValueError, match="kv must be"):
        zf.flash_attn_kvpacked_func(_bf16(1, 8, 4, 128), _bf16(1, 8, 3, 4, 128))


@pytest.mark.parametrize("kw", [{"softcap": 1.0}, {"alibi_slopes": torch.zeros(4)}])
def test_unsupported_features_raise(kw):
    with pytest.raises(ValueError, match="not supported"):
        zf.flash_attn_qkvpacked_func(_bf16(1, 8, 3, 4, 128), **kw)


def test_flash_attn_func_rejects_before_launch():
    q = _bf16(1, 8, 4, 128)
    with pytest.raises(ValueError, match="causal"):
        zf.flash_attn_func(q, q, q, causal=False)
    with pytest.raises(ValueError, match="sliding"):
        zf.flash_attn_func(q, q, q, window_size=(16, 0))
    with pytest.raises(TypeError, match="flash-attn 2's order"):
        zf.flash_attn_func(q, q, q, 0.1, True)  # flash-attn 3 positional order
    with pytest.raises(ValueError, match="layout"):
        zf.flash_attn_func(q, q, q, layout="sbhd")
    q8 = torch.zeros(1, 8, 4, 128, dtype=torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="descale"):
        zf.flash_attn_func(q8, q8, q8)


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
@pytest.mark.parametrize("want_lse", [False, True])
def test_custom_op_fake_shapes(layout, want_lse):
    with FakeTensorMode():
        if layout == "bshd":
            q, k, v = _bf16(2, 300, 8, 192), _bf16(2, 300, 2, 192), _bf16(2, 300, 2, 128)
            o_shape = (2, 300, 8, 128)
        else:
            q, k, v = _bf16(2, 8, 300, 192), _bf16(2, 2, 300, 192), _bf16(2, 2, 300, 128)
            o_shape = (2, 8, 300, 128)
        out, lse = torch.ops.zyfa.fwd(q, k, v, None, None, None, 0.07, layout, want_lse)
        assert tuple(out.shape) == o_shape and out.dtype == torch.bfloat16
        assert tuple(lse.shape) == ((2, 8, 300) if want_lse else (0,))
        assert lse.dtype == torch.float32
