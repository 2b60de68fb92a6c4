"""zyfa_fp8_quantize_noalloc: the quantiser entry point that allocates nothing.

Some callers cannot allocate device memory: code that is handed only the
buffers a host framework planned for it (a fixed memory arena, a plugin
interface that passes inputs and outputs and nothing else), or code on a path
where an allocation could stall the device.  For them the library keeps the
quantiser's small scratch (one maximum per CTA of the first pass) in a device
array of its own.  This test calls that entry point through the C ABI twice
in a row and checks each result against the workspace entry point, byte for
byte (the quantiser's outputs are e4m3 codes and a power-of-two descale, so
the tolerance is exact equality).  It lives in a file collected last and
builds and loads the library itself, so it passes alone in a fresh process
and after the other tests.
"""

import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    return zf.load()


def _quantize_with_workspace(x, xt, stream):
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    ds = torch.empty(1, dtype=torch.float32, device=x.device)
    ws = torch.empty(zf.zyfa_fp8_quantize_workspace_bytes(), dtype=torch.uint8, device=x.device)
    assert zf.zyfa_fp8_quantize(x.data_ptr(), x.numel(), xt, x8.data_ptr(), ds.data_ptr(),
                                ws.data_ptr(), stream) == zf.ZYFA_OK
    return x8, ds


def _quantize_without_allocation(x, xt, stream):
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    ds = torch.empty(1, dtype=torch.float32, device=x.device)
    assert zf.zyfa_fp8_quantize_noalloc(x.data_ptr(), x.numel(), xt, x8.data_ptr(),
                                        ds.data_ptr(), stream) == zf.ZYFA_OK
    return x8, ds


@pytest.mark.parametrize("dtype,xt", [(torch.bfloat16, zf.ZYFA_BF16),
                                      (torch.float32, zf.ZYFA_F32)])
def test_noalloc_matches_workspace_entry_point(lib, dtype, xt):
    stream = torch.cuda.current_stream().cuda_stream
    # Two different tensors back to back: the second call must not see the
    # first call's maxima (the shared array keeps the last call's contents).
    inputs = [(workloads.gaussian((3, 1000, 777), 901) * 40.0).to(dtype).cuda(),
              (workloads.gaussian((5, 333), 902) * 0.01).to(dtype).cuda()]
    for x in inputs:
        ref8, refds = _quantize_with_workspace(x, xt, stream)
        got8, gotds = _quantize_without_allocation(x, xt, stream)
        torch.cuda.synchronize()
        assert torch.equal(got8, ref8)
        assert torch.equal(gotds, refds)


def test_noalloc_rejects_bad_arguments(lib):
    assert zf.zyfa_fp8_quantize_noalloc(0, 16, zf.ZYFA_BF16, 0x10000, 0x10000, 0) == zf.ZYFA_ERR_ARG
    assert zf.zyfa_fp8_quantize_noalloc(0x10000, 16, zf.ZYFA_FP8_E4M3, 0x10000, 0x10000,
                                        0) == zf.ZYFA_ERR_UNSUPPORTED
