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

// Exponent k of the descale 2^k: the smallest power of two with
// amax / 2^k <= 448 (k = 0 for an all-zero tensor).  amax = f * 2^e with f in
// [0.5, 1): amax <= 448 * 2^k  <=>  f * 2^e <= 0.875 * 2^(k+9), so k = e - 9
// when f <= 0.875 and e - 8 otherwise.
__device__ __forceinline__ int descale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  const float f = frexpf(amax, &e);
  return e - 9 + (f > 0.875f ? 1 : 0);
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
    const int k = descale_exponent(m);
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

// ---------------------------------------------------------------------------
// Rotation before quantisation (ZYFA README, "Using FP8 attention in a
// model"): each row of d channels becomes x @ R, R = diag(s) H / sqrt(d) for
// d = 128 (H: Sylvester's Hadamard matrix) and R = diag(s) (C3^T kron H_64) / 8
// for d = 192 (C3: orthonormal 3-point DCT-II), then the rotated tensor is
// quantised per tensor as above.  One thread per row: the row is loaded into
// registers, multiplied by the signs (kept in shared memory), and transformed
// by in-register butterflies (H_2n = [[H_n, H_n], [H_n, -H_n]]: at stride h,
// channel pairs (i, i + h) with bit h of i clear become (a + b, a - b)); for
// d = 192 each 64-channel block is transformed and the three blocks are mixed
// by the DCT.  The first pass keeps max |x @ R|, the second recomputes the
// rotation and stores the codes (16 per 16-byte store).

constexpr int kRotThreads = 128;
constexpr int kRotRowsPerCta = kRotThreads / 2;

// Two lanes per row: lane half p = lane & 1 holds, for d = 128, channels
// 64p .. 64p+63 (local index i -> channel 64p + i); for d = 192, channels
// 64a + 32p .. 64a + 32p + 31 of each block a (local index 32a + i).  Every
// butterfly stride but the largest of each Hadamard block stays inside the
// lane; the largest (64 for d = 128, 32 for the 64-channel blocks of d = 192)
// pairs the two lanes of the row (shuffle distance 1).
template <int D>
struct RotHalf {
  static constexpr int kVals = D / 2;
  static constexpr int kBlock = D == 128 ? 64 : 32;  // contiguous channels per lane segment
  static __device__ __forceinline__ int channel(int i, int p) {
    return D == 128 ? 64 * p + i : 64 * (i / 32) + 32 * p + (i % 32);
  }
};

// Coalesced loads: a warp copies its 16 rows (contiguous in memory) into
// shared memory with consecutive 16-byte chunks per lane, laid out by lane
// (row r, half p -> lane 2r + p) with 16 bytes of padding per lane so that
// the lanes' reads of their own halves hit distinct banks; then each lane
// converts its half to FP32.
template <int D, int XT>
struct RotStage {
  static constexpr int kElem = XT == kQuantBF16 ? 2 : 4;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kHalfBytes = kRowBytes / 2;
  static constexpr int kPitch = kHalfBytes + 16;
  static constexpr int kWarpBytes = 32 * kPitch;
  static_assert(kHalfBytes % 16 == 0 && (D == 128 || (kRowBytes / 6) % 16 == 0), "16-byte chunks");
};

template <int D, int XT>
__device__ __forceinline__ void rot_stage_load(const void* x, int64_t row0, int64_t rows,
                                               uint8_t* wsm, int lane, float (&v)[D / 2]) {
  using T = RotStage<D, XT>;
  constexpr int kChunksPerRow = T::kRowBytes / 16;
  const uint8_t* src = static_cast<const uint8_t*>(x) + row0 * T::kRowBytes;
  __syncwarp();  // the previous rows have been read out
#pragma unroll 4
  for (int c = lane; c < 16 * kChunksPerRow; c += 32) {
    const int r = c / kChunksPerRow;
    const int off = (c % kChunksPerRow) * 16;
    if (row0 + r >= rows) continue;
    int half, local;
    if constexpr (D == 128) {
      half = off / T::kHalfBytes;
      local = off % T::kHalfBytes;
    } else {
      constexpr int kSeg = T::kRowBytes / 3;   // one 64-channel block
      const int a = off / kSeg, pos = off % kSeg;
      half = pos / (kSeg / 2);
      local = a * (kSeg / 2) + pos % (kSeg / 2);
    }
    *reinterpret_cast<uint4*>(wsm + (2 * r + half) * T::kPitch + local) =
        *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(c) * 16);
  }
  __syncwarp();
  const uint4* mine = reinterpret_cast<const uint4*>(wsm + lane * T::kPitch);
#pragma unroll
  for (int j = 0; j < T::kHalfBytes / 16; ++j) {
    const uint4 w = mine[j];
    if constexpr (XT == kQuantBF16) {
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[8 * j + 2 * k] = __uint_as_float(u[k] << 16);
        v[8 * j + 2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
      }
    } else {
      v[4 * j] = __uint_as_float(w.x); v[4 * j + 1] = __uint_as_float(w.y);
      v[4 * j + 2] = __uint_as_float(w.z); v[4 * j + 3] = __uint_as_float(w.w);
    }
  }
}

// In-register Hadamard butterflies of strides 1 .. n/2 on n channels at v[o].
// Strides of 2 and more pair neighbouring channels, so two butterflies run as
// one FP32x2 add and one FP32x2 multiply-add by -1 (exact: a - b rounded once).
template <int N, int M>
__device__ __forceinline__ void fwht_local(float (&v)[M], int o) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float a = v[o + i], b = v[o + i + 1];
    v[o + i] = a + b;
    v[o + i + 1] = a - b;
  }
  const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 2; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      if (i & h) continue;
      const float2 a = make_float2(v[o + i], v[o + i + 1]);
      const float2 b = make_float2(v[o + i + h], v[o + i + h + 1]);
      const float2 sum = __fadd2_rn(a, b);
      const float2 dif = __ffma2_rn(b, neg1, a);
      v[o + i] = sum.x; v[o + i + 1] = sum.y;
      v[o + i + h] = dif.x; v[o + i + h + 1] = dif.y;
    }
  }
}

// The butterfly stride that pairs the two lanes of a row: the lower half
// keeps a + b, the upper a - b, i.e. v' = v * (+1 or -1) + partner, exactly
// (one rounding), two channels per FP32x2 multiply-add.
template <int N>
__device__ __forceinline__ void cross_half(float (&v)[N], int p) {
  const float sgn = p ? -1.0f : 1.0f;
  const float2 s2 = make_float2(sgn, sgn);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float o0 = __shfl_xor_sync(0xffffffffu, v[i], 1);
    const float o1 = __shfl_xor_sync(0xffffffffu, v[i + 1], 1);
    const float2 r = __ffma2_rn(make_float2(v[i], v[i + 1]), s2, make_float2(o0, o1));
    v[i] = r.x;
    v[i + 1] = r.y;
  }
}

// x @ R of the row, this lane's half, in place (s_signs: D signs in shared
// memory, stored as [p][D/2 + 1] so that the two halves use different banks).
// Adding +0 at the end makes an exactly zero result +0 (its sign would
// otherwise depend on the order of the sums), so a zero always gets code 0x00.
template <int D>
__device__ __forceinline__ void rot_half(float (&v)[D / 2], const float* s_signs, int p) {
  constexpr int kN = D / 2;
  const float* sg = s_signs + p * (kN + 1);
#pragma unroll
  for (int i = 0; i < kN; i += 2) {
    const float2 r = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(sg[i], sg[i + 1]));
    v[i] = r.x;
    v[i + 1] = r.y;
  }
  if constexpr (D == 128) {
    fwht_local<64>(v, 0);
    cross_half<64>(v, p);
    constexpr float kScale = 0.08838834764831845f;  // 1 / sqrt(128)
    const float2 sc = make_float2(kScale, kScale), zero = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const float2 r = __ffma2_rn(make_float2(v[i], v[i + 1]), sc, zero);
      v[i] = r.x;
      v[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int a = 0; a < 3; ++a) fwht_local<32>(v, 32 * a);
    cross_half<96>(v, p);
    constexpr float kR3 = 0.57735026918962576f * 0.125f;   // 1/sqrt(3) / 8
    constexpr float kR2 = 0.70710678118654752f * 0.125f;   // 1/sqrt(2) / 8
    constexpr float kR6 = 0.40824829046386302f * 0.125f;   // 1/sqrt(6) / 8
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float b0 = v[e], b1 = v[32 + e], b2 = v[64 + e];
      v[e] = (b0 + b1 + b2) * kR3 + 0.0f;
      v[32 + e] = (b0 - b2) * kR2 + 0.0f;
      v[64 + e] = (b0 - 2.0f * b1 + b2) * kR6 + 0.0f;
    }
  }
}

template <int D>
__device__ __forceinline__ void rot_signs_to_smem(const float* signs, float* s_signs) {
  constexpr int kN = D / 2;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    // channel c -> (half p, local index i)
    int p, i;
    if (D == 128) {
      p = c / 64;
      i = c % 64;
    } else {
      p = (c % 64) / 32;
      i = 32 * (c / 64) + c % 32;
    }
    s_signs[p * (kN + 1) + i] = signs[c];
  }
}

template <int D, int XT>
__global__ void __launch_bounds__(kRotThreads)
    rot_amax_kernel(const void* x, int64_t rows, const float* signs, float* partial) {
  __shared__ float s_signs[D + 2];
  __shared__ float warp_max[kRotThreads / 32];
  rot_signs_to_smem<D>(signs, s_signs);
  __syncthreads();
  const int p = threadIdx.x & 1;
  const int lane = threadIdx.x & 31;
  extern __shared__ __align__(16) uint8_t rot_smem[];
  uint8_t* wsm = rot_smem + (threadIdx.x >> 5) * RotStage<D, XT>::kWarpBytes;
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRotRowsPerCta;
  // a warp takes 16 consecutive rows per iteration (row = row0 + lane / 2);
  // the loop condition is warp-uniform
  for (int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRotRowsPerCta + (threadIdx.x >> 5) * 16;
       row0 < rows; row0 += stride) {
    float v[D / 2];
    const bool live = row0 + (lane >> 1) < rows;
    rot_stage_load<D, XT>(x, row0, rows, wsm, lane, v);
    if (!live) {
#pragma unroll
      for (int i = 0; i < D / 2; ++i) v[i] = 0.f;
    }
    rot_half<D>(v, s_signs, p);
#pragma unroll
    for (int i = 0; i < D / 2; ++i) m = fmaxf(m, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 0.f;
    for (int i = 0; i < kRotThreads / 32; ++i) r = fmaxf(r, warp_max[i]);
    partial[blockIdx.x] = r;
  }
}

template <int D, int XT>
__global__ void __launch_bounds__(kRotThreads)
    rot_quant_kernel(const void* x, int64_t rows, const float* signs, uint8_t* x8,
                     float* descale, const float* partial, int num_partials) {
  __shared__ float s_signs[D + 2];
  __shared__ float warp_max[kRotThreads / 32];
  __shared__ float s_inv;
  float m = 0.f;
  for (int i = threadIdx.x; i < num_partials; i += kRotThreads) m = fmaxf(m, partial[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  rot_signs_to_smem<D>(signs, s_signs);
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 0.f;
    for (int i = 0; i < kRotThreads / 32; ++i) r = fmaxf(r, warp_max[i]);
    const int k = descale_exponent(r);
    s_inv = ldexpf(1.0f, -k);
    if (blockIdx.x == 0) *descale = ldexpf(1.0f, k);
  }
  __syncthreads();
  const float inv = s_inv;
  const int p = threadIdx.x & 1;
  constexpr int kSeg = RotHalf<D>::kBlock;
  constexpr int kSegs = (D / 2) / kSeg;
  const int lane = threadIdx.x & 31;
  extern __shared__ __align__(16) uint8_t rot_smem[];
  uint8_t* wsm = rot_smem + (threadIdx.x >> 5) * RotStage<D, XT>::kWarpBytes;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRotRowsPerCta;
  for (int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRotRowsPerCta + (threadIdx.x >> 5) * 16;
       row0 < rows; row0 += stride) {
    float v[D / 2];
    const int64_t row = row0 + (lane >> 1);
    const bool live = row < rows;
    rot_stage_load<D, XT>(x, row0, rows, wsm, lane, v);
    if (!live) {
#pragma unroll
      for (int i = 0; i < D / 2; ++i) v[i] = 0.f;
    }
    rot_half<D>(v, s_signs, p);
    if (live) {
#pragma unroll
      for (int g = 0; g < kSegs; ++g) {
        uint4* dst = reinterpret_cast<uint4*>(x8 + row * D + RotHalf<D>::channel(g * kSeg, p));
#pragma unroll
        for (int j = 0; j < kSeg / 16; ++j) {
          const float* w = v + g * kSeg + 16 * j;
          uint4 o;
          o.x = e4m3x4(w[0] * inv, w[1] * inv, w[2] * inv, w[3] * inv);
          o.y = e4m3x4(w[4] * inv, w[5] * inv, w[6] * inv, w[7] * inv);
          o.z = e4m3x4(w[8] * inv, w[9] * inv, w[10] * inv, w[11] * inv);
          o.w = e4m3x4(w[12] * inv, w[13] * inv, w[14] * inv, w[15] * inv);
          dst[j] = o;
        }
      }
    }
  }
}

int rot_grid(int64_t rows, int cap) {
  const int64_t want = (rows + kRotRowsPerCta - 1) / kRotRowsPerCta;
  if (want < 1) return 1;
  return want < cap ? static_cast<int>(want) : cap;
}

template <int D, int XT>
int launch_rot_t(const void* x, int64_t rows, const float* signs, void* x8, float* descale,
                 float* partial, int sms, cudaStream_t s) {
  const int g1 = rot_grid(rows, kQuantMaxPartials < 4 * sms ? kQuantMaxPartials : 4 * sms);
  constexpr int kSmem = (kRotThreads / 32) * RotStage<D, XT>::kWarpBytes;
  cudaError_t e = cudaFuncSetAttribute(rot_amax_kernel<D, XT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(rot_quant_kernel<D, XT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmem);
  if (e != cudaSuccess) return e;
  rot_amax_kernel<D, XT><<<g1, kRotThreads, kSmem, s>>>(x, rows, signs, partial);
  const int g2 = rot_grid(rows, 8 * sms);
  rot_quant_kernel<D, XT><<<g2, kRotThreads, kSmem, s>>>(x, rows, signs,
                                                         static_cast<uint8_t*>(x8), descale,
                                                         partial, g1);
  return cudaGetLastError();
}

}  // namespace

int launch_fp8_quantize(const void* x, int64_t n, int x_type, void* x8, float* descale,
                        float* partial, int sms, cudaStream_t stream) {
  if (x_type == kQuantBF16) return launch_t<kQuantBF16>(x, n, x8, descale, partial, sms, stream);
  if (x_type == kQuantF32) return launch_t<kQuantF32>(x, n, x8, descale, partial, sms, stream);
  return cudaErrorInvalidValue;
}

int launch_fp8_quantize_rotated(const void* x, int64_t rows, int d, int x_type,
                                const float* signs, void* x8, float* descale, float* partial,
                                int sms, cudaStream_t stream) {
  if (d == 128 && x_type == kQuantBF16)
    return launch_rot_t<128, kQuantBF16>(x, rows, signs, x8, descale, partial, sms, stream);
  if (d == 128 && x_type == kQuantF32)
    return launch_rot_t<128, kQuantF32>(x, rows, signs, x8, descale, partial, sms, stream);
  if (d == 192 && x_type == kQuantBF16)
    return launch_rot_t<192, kQuantBF16>(x, rows, signs, x8, descale, partial, sms, stream);
  if (d == 192 && x_type == kQuantF32)
    return launch_rot_t<192, kQuantF32>(x, rows, signs, x8, descale, partial, sms, stream);
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
