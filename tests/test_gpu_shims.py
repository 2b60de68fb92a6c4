"""The flash-attn style wrappers on the GPU: the packed and equal-length varlen
forms give bit-for-bit the result of ``flash_attn_func`` on the same tensors
(one of them also checked against the oracle), calls traced by torch.compile
and captured in a CUDA graph reproduce the eager result exactly, and backward
raises."""

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads
from gpu_util import assert_parity, run_oracle

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()
    torch.cuda.init()


def _gauss(shape, seed, dtype=torch.bfloat16):
    return workloads.gaussian(shape, seed).to(dtype).cuda()


def _fp8(shape, seed):
    x8, ds = zf.fp8_quantize(workloads.gaussian(shape, seed).cuda())
    return x8, ds


def test_qkvpacked_matches_oracle_and_unpacked():
    w = W["bf16_mha_b1_h2_s256_d128"]
    t = workloads.make_inputs(w)
    qkv = torch.stack([t["q"], t["k"], t["v"]], dim=2).cuda()   # (B, S, 3, H, d)
    out, lse = zf.flash_attn_qkvpacked_func(qkv, causal=True, return_lse=True)
    ref, ref_lse = zf.flash_attn_func(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], causal=True,
                                      return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    O, L = out.float().cpu().double().numpy(), lse.cpu().double().numpy()
    Oref, Lref = run_oracle(t, w)
    assert_parity(O, L, Oref, Lref, "bf16", "qkvpacked")


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_kvpacked_gqa_matches_unpacked(dt):
    B, S, H, Hkv, d = 2, 300, 8, 2, 128
    if dt == "bf16":
        q, kv = _gauss((B, S, H, d), 11), _gauss((B, S, 2, Hkv, d), 12)
        kw = {}
    else:
        (q, qs), (kv, kvs) = _fp8((B, S, H, d), 11), _fp8((B, S, 2, Hkv, d), 12)
        kw = dict(q_descale=qs, k_descale=kvs, v_descale=kvs)
    out = zf.flash_attn_kvpacked_func(q, kv, causal=True, **kw)
    ref = zf.flash_attn_func(q, kv[:, :, 0], kv[:, :, 1], causal=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("S", [256, 333])
def test_varlen_equal_lengths_match_batched(S):
    B, H, Hkv, d = 3, 4, 2, 128
    q, k, v = _gauss((B * S, H, d), 21), _gauss((B * S, Hkv, d), 22), _gauss((B * S, Hkv, d), 23)
    cu = torch.arange(0, B * S + 1, S, dtype=torch.int32, device="cuda")
    out, lse = zf.flash_attn_varlen_func(q, k, v, cu, cu, S, S, causal=True, return_lse=True)
    ref, ref_lse = zf.flash_attn_func(q.view(B, S, H, d), k.view(B, S, Hkv, d),
                                      v.view(B, S, Hkv, d), causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert out.shape == (B * S, H, d) and lse.shape == (H, B * S)
    assert torch.equal(out, ref.view(B * S, H, d))
    assert torch.equal(lse, ref_lse.permute(1, 0, 2).reshape(H, B * S))


def test_torch_compile_traces_through():
    q, k, v = _gauss((1, 640, 8, 128), 31), _gauss((1, 640, 2, 128), 32), _gauss((1, 640, 2, 128), 33)

    def f(q, k, v):
        out, lse = zf.flash_attn_func(q, k, v, causal=True, return_lse=True)
        return out, lse

    compiled = torch.compile(f, backend="aot_eager", fullgraph=True)
    out_c, lse_c = compiled(q, k, v)
    out_e, lse_e = f(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(out_c, out_e) and torch.equal(lse_c, lse_e)


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_cuda_graph_capture_replays_exactly(dt):
    shape_q, shape_kv = (1, 700, 8, 128), (1, 700, 2, 128)
    if dt == "bf16":
        q, k, v = _gauss(shape_q, 41), _gauss(shape_kv, 42), _gauss(shape_kv, 43)
        kw = {}
    else:
        (q, qs), (k, ks), (v, vs) = _fp8(shape_q, 41), _fp8(shape_kv, 42), _fp8(shape_kv, 43)
        kw = dict(q_descale=qs, k_descale=ks, v_descale=vs)
    eager = zf.flash_attn_func(q, k, v, causal=True, **kw)  # first call outside the capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            captured = zf.flash_attn_func(q, k, v, causal=True, **kw)
    torch.cuda.current_stream().wait_stream(s)
    captured.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(captured, eager)
    # new inputs in the same buffers flow through the replay
    q.copy_(_gauss(shape_q, 44) if dt == "bf16" else _fp8(shape_q, 44)[0])
    g.replay()
    fresh = zf.flash_attn_func(q, k, v, causal=True, **kw)
    torch.cuda.synchronize()
    assert torch.equal(captured, fresh)


def test_backward_raises():
    q = _gauss((1, 128, 2, 128), 51).requires_grad_(True)
    k, v = _gauss((1, 128, 2, 128), 52), _gauss((1, 128, 2, 128), 53)
    out = zf.flash_attn_func(q, k, v, causal=True)
    assert out.requires_grad
    with pytest.raises(RuntimeError, match="no backward"):
        out.float().sum().backward()
