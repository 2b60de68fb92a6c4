// Per-tensor FP8 e4m3 quantisation with a power-of-two descale: the input
// preparation step of the FP8 path (ZYFA README, "Usage": fp8_quantize
// returns the e4m3 tensor and one power-of-two descale per tensor, as a GPU
// scalar so that no call waits for the host; "Kernel design": every
// conversion rounds to nearest even).
//
// descale = smallest power of two with max|x| / descale <= 448 (1 for an
// all-zero tensor); x8 = e4m3_rne_satfinite(x / descale).
//
// Two deterministic passes (no atomics):
//   1. amax_kernel: each CTA writes the maximum |x| of its grid-stride share
//      to partial[blockIdx.x] (the workspace);
//   2. quant_kernel: every CTA reduces all partials (a few hundred floats),
//      derives the descale exactly from the exponent and mantissa of the
//      maximum, and converts its share; CTA 0 stores the descale.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "quant.h"

namespace zyfa {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;  // elements per thread per step

// Eight consecutive input elements as floats (BF16: one 16-byte load;
// FP32: two).
template <int XT>
__device__ __forceinline__ void load8(const void* x, int64_t i, float (&v)[8]) {
  if constexpr (XT == kQuantBF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + i);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(u[k] << 16);
      v[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + i);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + i + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <int XT>
__device__ __forceinline__ float load1(const void* x, int64_t i) {
  if constexpr (XT == kQuantBF16)
    return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[i]);
  else
    return static_cast<const float*>(x)[i];
}

__device__ __forceinline__ float block_max(float m) {
  __shared__ float warp_max[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kThreads / 32 ? warp_max[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  }
  return m;  // valid in warp 0
}

template <int XT>
__global__ void __launch_bounds__(kThreads) amax_kernel(const void* x, int64_t n, float* partial) {
  float m = 0.f;
  const int64_t nvec = n / kVec;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < nvec; v += stride) {
    float e[8];
    load8<XT>(x, v * kVec, e);
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(e[k]));
  }
  if (blockIdx.x == 0)
    for (int64_t i = nvec * kVec + threadIdx.x; i < n; i += kThreads) m = fmaxf(m, fabsf(load1<XT>(x, i)));
  m = block_max(m);
  if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

// Four FP32 -> four e4m3 bytes (byte k = value k), round to nearest even,
// saturating to +-448.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

__device__ __forceinline__ uint8_t e4m3x1(float a) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(a));
  return static_cast<uint8_t>(r & 0xFF);
}

template <int XT>
__global__ void __launch_bounds__(kThreads)
    quant_kernel(const void* x, int64_t n, uint8_t* x8, float* descale, const float* partial,
                 int num_partials) {
  __shared__ float s_inv;
  float m = 0.f;
  for (int i = threadIdx.x; i < num_partials; i += kThreads) m = fmaxf(m, partial[i]);
  m = block_max(m);
  if (threadIdx.x == 0) {
    // amax = f * 2^e with f in [0.5, 1): amax <= 448 * 2^k  <=>  f * 2^e <= 0.875 * 2^(k+9),
    // so k = e - 9 when f <= 0.875 and e - 8 otherwise.
    int k = 0;
    if (m > 0.f) {
      int e;
      const float f = frexpf(m, &e);
      k = e - 9 + (f > 0.875f ? 1 : 0);
    }
    s_inv = ldexpf(1.0f, -k);
    if (blockIdx.x == 0) *descale = ldexpf(1.0f, k);
  }
  __syncthreads();
  const float inv = s_inv;
  const int64_t nvec = n / kVec;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < nvec; v += stride) {
    float e[8];
    load8<XT>(x, v * kVec, e);
    uint2 o;
    o.x = e4m3x4(e[0] * inv, e[1] * inv, e[2] * inv, e[3] * inv);
    o.y = e4m3x4(e[4] * inv, e[5] * inv, e[6] * inv, e[7] * inv);
    *reinterpret_cast<uint2*>(x8 + v * kVec) = o;
  }
  if (blockIdx.x == 0)
    for (int64_t i = nvec * kVec + threadIdx.x; i < n; i += kThreads) x8[i] = e4m3x1(load1<XT>(x, i) * inv);
}

int grid_for(int64_t n, int cap) {
  const int64_t want = (n / kVec + kThreads - 1) / kThreads;
  if (want < 1) return 1;
  return want < cap ? static_cast<int>(want) : cap;
}

template <int XT>
int launch_t(const void* x, int64_t n, void* x8, float* descale, float* partial, int sms,
             cudaStream_t s) {
  const int g1 = grid_for(n, kQuantMaxPartials < 4 * sms ? kQuantMaxPartials : 4 * sms);
  amax_kernel<XT><<<g1, kThreads, 0, s>>>(x, n, partial);
  const int g2 = grid_for(n, 8 * sms);
  quant_kernel<XT><<<g2, kThreads, 0, s>>>(x, n, static_cast<uint8_t*>(x8), descale, partial, g1);
  return cudaGetLastError();
}

}  // namespace

int launch_fp8_quantize(const void* x, int64_t n, int x_type, void* x8, float* descale,
                        float* partial, int sms, cudaStream_t stream) {
  if (x_type == kQuantBF16) return launch_t<kQuantBF16>(x, n, x8, descale, partial, sms, stream);
  if (x_type == kQuantF32) return launch_t<kQuantF32>(x, n, x8, descale, partial, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zyfa

// ---------------------------------------------------------------------------
// Variant without a caller workspace, for callers that cannot allocate device
// memory: the per-CTA maxima of the first pass go to a file-scope array
// instead.  Every device that loads this library keeps these 4 KB until the
// process exits, and every call on a device shares them.
// ---------------------------------------------------------------------------
#include <mutex>

namespace zyfa {
namespace {

static __device__ __align__(256) float g_noalloc_partials[kQuantMaxPartials];

constexpr int kMaxDevicesNoAlloc = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevicesNoAlloc] = {};

}  // namespace

int fp8_quantize_noalloc(const void* x, int64_t n, int x_type, void* x8, float* descale, int sms,
                         cudaStream_t stream, int* too_large) {
  *too_large = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesNoAlloc) return cudaErrorInvalidDevice;
  float* partials = nullptr;
  {
    // One-time set-up per device, with that device current: host code needs
    // the array's device address (its name is only a host-side stand-in).
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_partials);
      if (e != cudaSuccess) return e;
      g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    partials = g_noalloc_ptr[dev];
  }
  // The first pass writes one maximum per CTA and launches at most
  // min(kQuantMaxPartials, 4 * SMs) CTAs; reject a device whose first pass
  // would need more slots than the array holds.
  const int slots = kQuantMaxPartials < 4 * sms ? kQuantMaxPartials : 4 * sms;
  if (slots > static_cast<int>(sizeof(g_noalloc_partials) / sizeof(float))) {
    *too_large = 1;
    return cudaErrorInvalidValue;
  }
  // Nothing needs clearing: the second pass reads only the slots the first
  // pass of the same call has written.
  return launch_fp8_quantize(x, n, x_type, x8, descale, partials, sms, stream);
}

}  // namespace zyfa
