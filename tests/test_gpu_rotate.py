"""Rotation + FP8 quantisation on the GPU against the float64 oracle.

The kernel rotates in FP32, the oracle in float64, so a code is compared only
where the decision is settled: the oracle's scaled value y/descale is widened
by a bound on the FP32 rotation error (row-wise, from the L1 norm of the row)
and every code whose e4m3 value lies between the codes of the two ends is
accepted; where both ends round to the same code (almost every element) the
code must match exactly.  The descale is checked the same way.  A rotated
value that is exactly zero is quantised to +0, and codes of zero are
compared without their sign (the sign of a value that rounds to zero depends
on the order of the sums)."""

import math

import numpy as np
import pytest
import torch

import causal_flashattention_prefill_gb300 as zf
import oracle
import workloads
from oracle.formats import e4m3_to_f64
from oracle.quantize import descale_of, e4m3_encode_rne

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from causal_flashattention_prefill_gb300 import build
    build.build()
    zf.load()
    torch.cuda.init()


def _check_against_oracle(x_host: np.ndarray, signs: np.ndarray, codes: np.ndarray, ds: float):
    d = x_host.shape[-1]
    xr = x_host.reshape(-1, d)
    y = oracle.rotate_f64(xr, signs)
    # FP32 rotation error: log2(d) + 3 roundings of partial sums bounded by the
    # row's L1 norm (scaled), plus the input scale constant; generous factor 4.
    stages = 8 if d == 128 else 10
    bound = 4.0 * stages * 2.0 ** -24 * np.abs(xr).sum(axis=1, keepdims=True) / math.sqrt(d)
    bound = np.broadcast_to(bound, y.shape)
    amax = np.abs(y).max()
    b_max = bound.max()
    assert ds in {descale_of(max(amax - b_max, 0.0)), descale_of(amax + b_max)}, (ds, amax)
    lo = e4m3_to_f64(e4m3_encode_rne((y - bound) / ds))
    hi = e4m3_to_f64(e4m3_encode_rne((y + bound) / ds))
    got = e4m3_to_f64(codes.reshape(y.shape))
    ok = (got >= np.minimum(lo, hi)) & (got <= np.maximum(lo, hi))
    assert ok.all(), f"{(~ok).sum()} codes outside the settled range"
    settled = lo == hi
    # zero is compared without its sign: a value that rounds to zero takes its
    # sign from the last rounding of the sums, which FP32 and float64 order
    # differently
    want = e4m3_encode_rne(y / ds)
    want = np.where(want == 0x80, 0, want)
    got_c = codes.reshape(y.shape)
    got_c = np.where(got_c == 0x80, 0, got_c)
    exact = np.array_equal(got_c[settled], want[settled])
    assert exact
    return settled.mean()


@pytest.mark.parametrize("d", [128, 192])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("rows,scale", [(1, 1.0), (7, 30.0), (1000, 0.01), (4099, 5.0)])
def test_rotated_quantize_matches_oracle(d, dt, rows, scale):
    x = (workloads.gaussian((rows, d), 700 + rows + d) * scale).to(dt)
    signs = zf.hadamard_signs(d, seed=rows)
    x8, ds = zf.fp8_quantize_rotated(x.cuda(), signs)
    torch.cuda.synchronize()
    codes = x8.view(torch.uint8).cpu().numpy()
    frac = _check_against_oracle(x.double().numpy(), signs.cpu().double().numpy(), codes,
                                 float(ds.item()))
    assert frac > 0.99


@pytest.mark.parametrize("d,dt", [(128, torch.bfloat16), (192, torch.float32)], ids=["d128-bf16", "d192-f32"])
def test_rotated_quantize_many_tiles_per_cta(d, dt):
    # more 64-row tiles than CTAs x ring stages, so every CTA's ring wraps
    # several times, with a ragged last tile
    rows = 140001 if d == 128 else 60017
    x = (workloads.gaussian((rows, d), 77 + d) * 2.0).to(dt)
    signs = zf.hadamard_signs(d, seed=11)
    x8, ds = zf.fp8_quantize_rotated(x.cuda(), signs)
    torch.cuda.synchronize()
    frac = _check_against_oracle(x.double().numpy(), signs.cpu().double().numpy(),
                                 x8.view(torch.uint8).cpu().numpy(), float(ds.item()))
    assert frac > 0.99


def test_rotated_quantize_zero_rows():
    # n_rows = 0 through the C ABI: descale 1, no code written, no wait timed out
    x = torch.ones(64, 128, dtype=torch.bfloat16, device="cuda")
    x8 = torch.full((64, 128), 0x55, dtype=torch.uint8, device="cuda")
    ds = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(zf.zyfa_fp8_quantize_workspace_bytes(), dtype=torch.uint8, device="cuda")
    signs = zf.hadamard_signs(128)
    st = zf.zyfa_fp8_quantize_rotated(x.data_ptr(), 0, 128, zf.ZYFA_BF16, signs.data_ptr(),
                                      x8.data_ptr(), ds.data_ptr(), ws.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == zf.ZYFA_OK and float(ds.item()) == 1.0
    assert int(x8.min()) == 0x55 and int(x8.max()) == 0x55
    assert zf.zyfa_device_status(reset=True) == (zf.ZYFA_OK, 0)


@pytest.mark.parametrize("d,rows", [(128, 4099), (192, 1001)])
def test_rotated_quantize_writes_only_its_rows(d, rows):
    # Codes are staged in shared memory and stored as whole rows: the call
    # writes exactly n_rows * d bytes (ragged last tile), equal to the shim's
    # codes, and leaves the bytes after them untouched.
    x = (workloads.gaussian((rows, d), 4242 + d) * 3.0).to(torch.bfloat16).cuda()
    signs = zf.hadamard_signs(d, seed=d)
    ref8, ref_ds = zf.fp8_quantize_rotated(x, signs)
    pad = 4096
    x8 = torch.full((rows * d + pad,), 0xA5, dtype=torch.uint8, device="cuda")
    ds = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(zf.zyfa_fp8_quantize_workspace_bytes(), dtype=torch.uint8, device="cuda")
    st = zf.zyfa_fp8_quantize_rotated(x.data_ptr(), rows, d, zf.ZYFA_BF16, signs.data_ptr(),
                                      x8.data_ptr(), ds.data_ptr(), ws.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == zf.ZYFA_OK and zf.zyfa_device_status(reset=True) == (zf.ZYFA_OK, 0)
    assert float(ds.item()) == float(ref_ds.item())
    assert torch.equal(x8[: rows * d], ref8.view(torch.uint8).reshape(-1))
    assert int(x8[rows * d:].min()) == 0xA5 and int(x8[rows * d:].max()) == 0xA5


def test_rotated_quantize_activation_like_and_zero():
    # outlier channels (the case rotation is for) and an all-zero tensor
    g = torch.Generator().manual_seed(5)
    x = torch.randn(3000, 128, generator=g)
    x[:, [3, 40, 77, 100]] *= 20.0
    signs = zf.hadamard_signs(128, seed=0)
    x8, ds = zf.fp8_quantize_rotated(x.to(torch.bfloat16).cuda(), signs)
    torch.cuda.synchronize()
    _check_against_oracle(x.to(torch.bfloat16).double().numpy(), signs.cpu().double().numpy(),
                          x8.view(torch.uint8).cpu().numpy(), float(ds.item()))
    z8, zs = zf.fp8_quantize_rotated(torch.zeros(64, 192, dtype=torch.bfloat16, device="cuda"),
                                     zf.hadamard_signs(192))
    torch.cuda.synchronize()
    assert float(zs.item()) == 1.0 and int(z8.view(torch.uint8).max()) == 0


@pytest.mark.parametrize("d,dt,rows", [(128, torch.bfloat16, 524288), (192, torch.bfloat16, 200003),
                                        (128, torch.float32, 262144), (192, torch.float32, 20000)],
                         ids=["d128-bf16", "d192-bf16", "d128-f32", "d192-f32"])
def test_rotated_quantize_is_deterministic(d, dt, rows):
    # Repeated calls give identical codes.  At 524288 rows of d = 128 BF16
    # (a four-stage ring of 16 KB tiles) an earlier form of the kernel wrote
    # a few wrong rows in most calls, which the smaller oracle cases missed.
    g = torch.Generator(device="cuda").manual_seed(rows + d)
    x = (torch.randn(rows, d, generator=g, device="cuda") * 3.0).to(dt)
    s = zf.hadamard_signs(d, seed=3)
    a8, ad = zf.fp8_quantize_rotated(x, s)
    for _ in range(8):
        b8, bd = zf.fp8_quantize_rotated(x, s)
        torch.cuda.synchronize()
        assert torch.equal(a8.view(torch.uint8), b8.view(torch.uint8)) and torch.equal(ad, bd)
    assert zf.zyfa_device_status(reset=True) == (zf.ZYFA_OK, 0)


def _rel_rms(a, b):
    return float(np.sqrt(((a - b) ** 2).sum() / (b ** 2).sum()))


@pytest.mark.parametrize("d", [128, 192])
def test_rotation_lowers_fp8_attention_error(d):
    """The README's use: rotate q and k (same signs), leave v, quantise, run
    FP8 attention; on activation-like q/k (per-channel scales and outlier
    channels) the output is closer to the unquantised float64 attention than
    without the rotation, and it still matches the oracle on the rotated
    quantised inputs within the FP8 tolerances."""
    B, S, H, Hkv = 1, 1024, 4, 2
    g = torch.Generator().manual_seed(40 + d)
    chan = torch.exp(torch.randn(d, generator=g) * 0.5)
    out_ch = torch.randperm(d, generator=g)[:4]
    chan[out_ch] *= 20.0
    q = torch.randn(B, S, H, d, generator=g) * chan * 0.3
    k = torch.randn(B, S, Hkv, d, generator=g) * chan * 0.3
    v = torch.randn(B, S, Hkv, 128, generator=g)
    qb, kb, vb = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    ref_o, _ = oracle.attention_f64(qb.double().numpy(), kb.double().numpy(),
                                    vb.double().numpy(), dtype="f64", layout="bshd", scale=scale)
    dev = torch.device("cuda")
    v8, vs = zf.fp8_quantize(vb.to(dev))
    errs = {}
    for rotate in (False, True):
        if rotate:
            s = zf.hadamard_signs(d, seed=0)
            q8, qs = zf.fp8_quantize_rotated(qb.to(dev), s)
            k8, ks = zf.fp8_quantize_rotated(kb.to(dev), s)
        else:
            q8, qs = zf.fp8_quantize(qb.to(dev))
            k8, ks = zf.fp8_quantize(kb.to(dev))
        out = zf.flash_attn_func(q8, k8, v8, causal=True, softmax_scale=scale,
                                 q_descale=qs, k_descale=ks, v_descale=vs)
        torch.cuda.synchronize()
        errs[rotate] = _rel_rms(out.float().cpu().double().numpy(), ref_o)
        if rotate:
            # parity of the attention itself on the rotated, quantised inputs
            t = {"q": q8.cpu(), "k": k8.cpu(), "v": v8.cpu(), "q_descale": float(qs.item()),
                 "k_descale": float(ks.item()), "v_descale": float(vs.item())}
            O8, L8 = oracle.attention_f64(*(workloads.codes(t[n]) for n in "qkv"), dtype="fp8",
                                          layout="bshd", scale=scale, q_descale=t["q_descale"],
                                          k_descale=t["k_descale"], v_descale=t["v_descale"])
            dO = np.abs(out.float().cpu().double().numpy() - O8)
            assert dO.max() <= 4e-2 and dO.mean() <= 4e-3
    print(f"d={d} rel RMS vs unquantised: plain {errs[False]:.3e} rotated {errs[True]:.3e}")
    assert errs[True] < errs[False]
