// Per-tensor FP8 e4m3 quantisation with a power-of-two descale: the input
// preparation step of the FP8 path (ZYFA README, "Usage": fp8_quantize
// returns the e4m3 tensor and one power-of-two descale per tensor, as a GPU
// scalar so that no call waits for the host; "Kernel design": all format
// conversions use round-half-to-even).
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
#include "zyfa_ptx.cuh"

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
// quantised per tensor as above.  The butterflies of H_2n = [[H_n, H_n],
// [H_n, -H_n]] run in registers: at stride h, channel pairs (i, i + h) with
// bit h of i clear become (a + b, a - b); for d = 192 each 64-channel block
// is transformed and the three blocks are mixed by the DCT.  The first pass
// keeps max |x @ R|, the second recomputes the rotation and stores the codes.
//
// Data movement: tiles of 64 rows stream through a ring of shared-memory
// stages filled by TMA from a two-dimensional tensor map over (channels,
// rows) with 128-byte swizzle, one box of 64 rows x 128 bytes per 128 bytes
// of the row.  Warps 0-3 rotate 16 rows of each tile (lane = row lane & 15,
// half lane >> 4); warp 4 issues the copies.  The eight lanes of a quarter
// warp read 16-byte chunks of eight consecutive rows, which the swizzle
// places in eight distinct bank groups, so the reads are conflict-free.

constexpr int kRotTileRows = 64;
constexpr int kRotConsumers = 4;                       // warps that rotate
constexpr int kRotThreads = 32 * (kRotConsumers + 1);  // + one producer warp
constexpr int kRotSmemTarget = 64 * 1024;              // ring bytes per CTA (at least two stages)
// L2 reuse between the passes: the first pass reads the last tiles of x
// (those it loads last, up to this many bytes) with an evict_last hint and
// the others with evict_first, and the second pass walks every CTA's tiles
// in reverse order, so its first reads find them in L2.
constexpr int64_t kRotL2KeepBytes = int64_t(88) << 20;

// Status word of these kernels (bit 0: a wait timed out).
__device__ int g_rot_status;

template <int D, int XT>
struct RotTile {
  static constexpr int kElem = XT == kQuantBF16 ? 2 : 4;
  static constexpr int kBoxElems = 128 / kElem;            // inner box extent
  static constexpr int kBoxes = D * kElem / 128;           // boxes per row
  static constexpr int kBoxBytes = kRotTileRows * 128;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStagesFit = kRotSmemTarget / kTileBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : (kStagesFit < 2 ? 2 : kStagesFit);
  static constexpr int kChunks = D * kElem / 2 / 16;       // 16-byte chunks of a half row
  static constexpr int kPerChunk = 16 / kElem;             // values per chunk
  static constexpr int kSmem = 1024 + kStages * kTileBytes + 2 * kStages * 8 + 16;
  static_assert(D * kElem % 128 == 0, "whole boxes per row");
  static_assert(kStages >= 2, "ring needs two stages");
};

// Lane half p of a row holds, for d = 128, channels 64p .. 64p+63 (local
// index i -> channel 64p + i); for d = 192, channels 64a + 32p .. 64a + 32p +
// 31 of each block a (local index 32a + i).  Every butterfly stride but the
// largest of each Hadamard block stays inside the lane; the largest (64 for
// d = 128, 32 for the 64-channel blocks of d = 192) pairs the two lanes of
// the row (shuffle distance 16).
template <int D>
struct RotHalf {
  static constexpr int kBlock = D == 128 ? 64 : 32;  // contiguous channels per lane segment
  static __device__ __forceinline__ int channel(int i, int p) {
    return D == 128 ? 64 * p + i : 64 * (i / 32) + 32 * p + (i % 32);
  }
};

// This lane's half of row r of a tile in shared memory (boxes of 64 rows x
// 128 bytes, 128-byte swizzle: chunk c of a box row r sits at chunk c ^ (r & 7)),
// converted to FP32.
template <int D, int XT>
__device__ __forceinline__ void rot_read_half(const uint8_t* tile, int r, int p,
                                              float (&v)[D / 2]) {
  using T = RotTile<D, XT>;
#pragma unroll
  for (int k = 0; k < T::kChunks; ++k) {
    const int byte = RotHalf<D>::channel(k * T::kPerChunk, p) * T::kElem;
    const int box = byte >> 7, c16 = (byte & 127) >> 4;
    const uint4 w = *reinterpret_cast<const uint4*>(tile + box * T::kBoxBytes + r * 128 +
                                                    ((c16 ^ (r & 7)) << 4));
    if constexpr (XT == kQuantBF16) {
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[8 * k + 2 * q] = __uint_as_float(u[q] << 16);
        v[8 * k + 2 * q + 1] = __uint_as_float(u[q] & 0xFFFF0000u);
      }
    } else {
      v[4 * k] = __uint_as_float(w.x); v[4 * k + 1] = __uint_as_float(w.y);
      v[4 * k + 2] = __uint_as_float(w.z); v[4 * k + 3] = __uint_as_float(w.w);
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

// The butterfly stride that pairs the two lanes of a row (lanes l and l ^ 16):
// the lower half keeps a + b, the upper a - b, i.e. v' = v * (+1 or -1) +
// partner, exactly (one rounding), two channels per FP32x2 multiply-add.
template <int N>
__device__ __forceinline__ void cross_half(float (&v)[N], int p) {
  const float sgn = p ? -1.0f : 1.0f;
  const float2 s2 = make_float2(sgn, sgn);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float o0 = __shfl_xor_sync(0xffffffffu, v[i], 16);
    const float o1 = __shfl_xor_sync(0xffffffffu, v[i + 1], 16);
    const float2 r = __ffma2_rn(make_float2(v[i], v[i + 1]), s2, make_float2(o0, o1));
    v[i] = r.x;
    v[i + 1] = r.y;
  }
}

// x @ R of the row up to one constant factor per 32-channel block
// (rot_scale), this lane's half, in place (s_signs: D signs in shared memory,
// stored as [p][D/2 + 1] so that the two halves use different banks).  The
// factor is applied by the passes: the max pass scales the maximum once
// (rounding is monotonic, so the scaled maximum is the maximum of the scaled
// values), the quantise pass folds it into the descale multiply (a power of
// two, so one rounding gives the same value as two).
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
  } else {
#pragma unroll
    for (int a = 0; a < 3; ++a) fwht_local<32>(v, 32 * a);
    cross_half<96>(v, p);
    // DCT rows (1, 1, 1), (1, 0, -1), (1, -2, 1) over the three blocks
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float b0 = v[e], b1 = v[32 + e], b2 = v[64 + e];
      v[e] = (b0 + b1) + b2;
      v[32 + e] = b0 - b2;
      v[64 + e] = (b0 - 2.0f * b1) + b2;
    }
  }
}

// BF16 input: this lane's half of row r rotated as rot_half does, with the
// butterfly stride that pairs the two lanes of the row taken first, on the
// raw BF16 words (Hadamard stages commute; only the FP32 rounding order
// differs).  The signs come as XOR masks (bit 15 / 31 flips the BF16 value
// in the low / high half of a word), so a shuffle of one 32-bit word moves
// two values across the lane pair.
template <int D>
__device__ __forceinline__ void rot_half_bf16(const uint8_t* tile, int r, int p,
                                              const uint32_t (&mask)[D / 4], float (&v)[D / 2]) {
  using T = RotTile<D, kQuantBF16>;
  const float sgn = p ? -1.0f : 1.0f;
  const float2 s2 = make_float2(sgn, sgn);
#pragma unroll
  for (int k = 0; k < T::kChunks; ++k) {
    const int byte = RotHalf<D>::channel(k * T::kPerChunk, p) * 2;
    const int box = byte >> 7, c16 = (byte & 127) >> 4;
    const uint4 w4 = *reinterpret_cast<const uint4*>(tile + box * T::kBoxBytes + r * 128 +
                                                     ((c16 ^ (r & 7)) << 4));
    const uint32_t u[4] = {w4.x ^ mask[4 * k], w4.y ^ mask[4 * k + 1], w4.z ^ mask[4 * k + 2],
                           w4.w ^ mask[4 * k + 3]};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, u[q], 16);
      // lower lane: own + partner; upper lane: partner - own
      const float2 mine = make_float2(__uint_as_float(u[q] << 16), __uint_as_float(u[q] & 0xFFFF0000u));
      const float2 other = make_float2(__uint_as_float(o << 16), __uint_as_float(o & 0xFFFF0000u));
      const float2 y = __ffma2_rn(mine, s2, other);
      v[8 * k + 2 * q] = y.x;
      v[8 * k + 2 * q + 1] = y.y;
    }
  }
  if constexpr (D == 128) {
    fwht_local<64>(v, 0);
  } else {
#pragma unroll
    for (int a = 0; a < 3; ++a) fwht_local<32>(v, 32 * a);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float b0 = v[e], b1 = v[32 + e], b2 = v[64 + e];
      v[e] = (b0 + b1) + b2;
      v[32 + e] = b0 - b2;
      v[64 + e] = (b0 - 2.0f * b1) + b2;
    }
  }
}

// XOR masks of the signs for this lane's half (see rot_half_bf16): word j
// covers local values 2j and 2j + 1.
template <int D>
__device__ __forceinline__ void rot_sign_masks(const float* s_signs, int p,
                                               uint32_t (&mask)[D / 4]) {
  constexpr int kN = D / 2;
  const float* sg = s_signs + p * (kN + 1);
#pragma unroll
  for (int j = 0; j < D / 4; ++j)
    mask[j] = (sg[2 * j] < 0.f ? 0x8000u : 0u) | (sg[2 * j + 1] < 0.f ? 0x80000000u : 0u);
}

// Codes are staged in shared memory, eight rows of a warp at a time (16-byte
// chunk c of row r at chunk rot_code_chunk(c, r) of that row), so that each
// global store writes 512 contiguous bytes.  The permutation keeps both the
// per-lane writes (row r, its half of the channels) and the linear read-back
// free of bank conflicts.
template <int D>
__device__ __forceinline__ int rot_code_chunk(int c, int r) {
  return D == 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
}

// The factor of local 32-value block a: 1/sqrt(128) for d = 128; for d = 192
// the DCT's row norms times 1/8 (H_64 / 8 is orthonormal).
template <int D>
__device__ __forceinline__ constexpr float rot_scale(int a) {
  if (D == 128) return 0.08838834764831845f;            // 1 / sqrt(128)
  return a == 0 ? 0.57735026918962576f * 0.125f          // 1/sqrt(3) / 8
                : a == 1 ? 0.70710678118654752f * 0.125f  // 1/sqrt(2) / 8
                         : 0.40824829046386302f * 0.125f; // 1/sqrt(6) / 8
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

// Waits with the whole warp (see the attention kernel's warp_wait): every
// lane observes the completed phase, so the TMA-written tile is visible to
// all of them.
__device__ __forceinline__ bool rot_warp_wait(uint32_t b, uint32_t parity, volatile int* abort,
                                              int lane) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(b, parity))) return true;
  int ok = 0;
  if (lane == 0) ok = ptx::mbar_wait(b, parity, abort, &g_rot_status, 1) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) (void)ptx::mbar_test(b, parity);
  return ok != 0;
}

// One pass over the tensor.  kQuant = false: each CTA writes max |x @ R| of
// its tiles to partial[blockIdx.x].  kQuant = true: every CTA reduces the
// num_partials maxima to the descale, CTA 0 stores it, and each row's codes
// are written to x8.  CTA b takes tiles b + i * gridDim.x, i ascending in
// the first pass and descending in the second.
template <int D, int XT, bool kQuant>
__global__ void __launch_bounds__(kRotThreads)
    rot_pass_kernel(const __grid_constant__ CUtensorMap tm, int64_t rows, const float* signs,
                    float* partial, uint8_t* x8, float* descale, int num_partials) {
  using T = RotTile<D, XT>;
  constexpr int NS = T::kStages;
  __shared__ float s_signs[D + 2];
  __shared__ float warp_max[kRotConsumers + 1];
  __shared__ float s_inv;
  constexpr int kRowChunks = D / 16;               // 16-byte code chunks per row
  constexpr int kStageChunks = 8 * kRowChunks;     // 8 rows staged per warp at a time
  __shared__ uint4 s_codes[kQuant ? kRotConsumers * kStageChunks : 1];
  extern __shared__ uint8_t rot_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(rot_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + NS * T::kTileBytes);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 2 * NS);
  const uint32_t bar0 = ptx::smem_u32(bars);
  auto full = [&](int st) { return bar0 + 8u * static_cast<uint32_t>(st); };
  auto empty = [&](int st) { return bar0 + 8u * static_cast<uint32_t>(NS + st); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      ptx::mbar_init(full(st), 1);
      ptx::mbar_init(empty(st), kRotConsumers);
    }
    *abort = 0;
    ptx::fence_barrier_init();
  }
  rot_signs_to_smem<D>(signs, s_signs);
  if constexpr (kQuant) {
    float m = 0.f;
    for (int i = threadIdx.x; i < num_partials; i += kRotThreads) m = fmaxf(m, partial[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) warp_max[warp] = m;
  }
  __syncthreads();
  if constexpr (kQuant) {
    if (threadIdx.x == 0) {
      float r = 0.f;
      for (int i = 0; i < kRotConsumers + 1; ++i) r = fmaxf(r, warp_max[i]);
      const int k = descale_exponent(r);
      s_inv = ldexpf(1.0f, -k);
      if (blockIdx.x == 0) *descale = ldexpf(1.0f, k);
    }
    __syncthreads();
  }
  const int64_t n_tiles = (rows + kRotTileRows - 1) / kRotTileRows;
  const int64_t n_mine =
      n_tiles > blockIdx.x ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  // k-th tile of this CTA (k counts ring uses in both roles).
  auto tile_of = [&](int64_t k) {
    return static_cast<int64_t>(blockIdx.x) + (kQuant ? n_mine - 1 - k : k) * gridDim.x;
  };

  if (warp == kRotConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tm);
      // The first pass leaves its last tiles of x in L2 for the second; the
      // second reads x for the last time.
      const uint64_t pol_first = ptx::policy_evict_first();
      const uint64_t pol_last = ptx::policy_evict_last();
      const int64_t keep_from = n_tiles - kRotL2KeepBytes / T::kTileBytes;
      uint32_t armed = 0, par = 0;  // bit st: armed at least once / parity of its last arming
      for (int64_t i = 0; i < n_mine; ++i) {
        const int64_t tile = tile_of(i);
        const uint64_t pol = (!kQuant && tile >= keep_from) ? pol_last : pol_first;
        const int st = static_cast<int>(i % NS);
        const uint32_t round = static_cast<uint32_t>(i / NS);
        if (!ptx::mbar_wait(empty(st), (round & 1u) ^ 1u, abort, &g_rot_status, 1)) break;
        ptx::mbar_arrive_expect_tx(full(st), T::kTileBytes);
        const uint32_t dst = ptx::smem_u32(ring + st * T::kTileBytes);
#pragma unroll
        for (int bx = 0; bx < T::kBoxes; ++bx)
          ptx::tma_load_2d(dst + bx * T::kBoxBytes, &tm, full(st), bx * T::kBoxElems,
                           static_cast<int>(tile * kRotTileRows), pol);
        armed |= 1u << st;
        par = (par & ~(1u << st)) | ((round & 1u) << st);
      }
      // Every copy issued lands before the CTA's shared memory is released.
      for (int st = 0; st < NS; ++st)
        if ((armed >> st) & 1u) ptx::mbar_drain(full(st), (par >> st) & 1u);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ rotation
    const int r = 16 * warp + (lane & 15);  // row within the tile
    const int p = lane >> 4;                // half of the row
    // BF16 at d = 128 takes the sign-mask path (rot_half_bf16); at d = 192
    // its 48 mask registers would cost a CTA per SM (measured slower).
    constexpr bool kMaskPath = XT == kQuantBF16 && D == 128;
    uint32_t mask[kMaskPath ? D / 4 : 1];
    if constexpr (kMaskPath) rot_sign_masks<D>(s_signs, p, mask);
    float m = 0.f;
    for (int64_t i = 0; i < n_mine; ++i) {
      const int64_t tile = tile_of(i);
      const int st = static_cast<int>(i % NS);
      if (!rot_warp_wait(full(st), static_cast<uint32_t>(i / NS) & 1u, abort, lane)) break;
      float v[D / 2];
      if constexpr (kMaskPath) {
        rot_half_bf16<D>(ring + st * T::kTileBytes, r, p, mask, v);
      } else {
        rot_read_half<D, XT>(ring + st * T::kTileBytes, r, p, v);
      }
      // The stage goes back to the tensor copies (async proxy) after these
      // generic-proxy reads: order them before the release.
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty(st));
      // Rows past the end read TMA's zero fill: they rotate to zero and
      // leave the maximum unchanged; their codes are not stored.
      if constexpr (!kMaskPath) rot_half<D>(v, s_signs, p);
      if constexpr (!kQuant) {
#pragma unroll
        for (int a = 0; a < D / 64; ++a) {
          float mb = 0.f;
#pragma unroll
          for (int k = 0; k < 32; k += 2) mb = ptx::max3(mb, fabsf(v[32 * a + k]), fabsf(v[32 * a + k + 1]));
          m = fmaxf(m, mb * rot_scale<D>(a));
        }
      } else {
        // Rows past the end are converted too (zeros) but not stored.
        const float inv = s_inv;
        const float2 zero = make_float2(0.0f, 0.0f);
        constexpr int kSeg = RotHalf<D>::kBlock;
        constexpr int kLaneChunks = D / 32;  // 16-byte code chunks of a half row
        uint4 oc[kLaneChunks];
#pragma unroll
        for (int g = 0; g < (D / 2) / kSeg; ++g) {
#pragma unroll
          for (int j = 0; j < kSeg / 16; ++j) {
            // y = t * (factor * inv) + 0 (adding +0 makes an exactly zero
            // result +0, whose sign would otherwise follow the order of the
            // sums, so a zero always gets code 0x00)
            const int i0 = g * kSeg + 16 * j;
            const float c = rot_scale<D>(i0 / 32) * inv;
            const float2 c2 = make_float2(c, c);
            float y[16];
#pragma unroll
            for (int q = 0; q < 16; q += 2) {
              const float2 r = __ffma2_rn(make_float2(v[i0 + q], v[i0 + q + 1]), c2, zero);
              y[q] = r.x;
              y[q + 1] = r.y;
            }
            uint4& o = oc[i0 / 16];
            o.x = e4m3x4(y[0], y[1], y[2], y[3]);
            o.y = e4m3x4(y[4], y[5], y[6], y[7]);
            o.z = e4m3x4(y[8], y[9], y[10], y[11]);
            o.w = e4m3x4(y[12], y[13], y[14], y[15]);
          }
        }
        // Two rounds of 8 rows: the lanes of those rows write their chunks,
        // then the warp stores the rows with 512-byte contiguous writes.
        uint4* codes = s_codes + warp * kStageChunks;
        const int rw = lane & 15;  // row within the warp's 16 rows
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if ((rw >> 3) == h) {
#pragma unroll
            for (int k = 0; k < kLaneChunks; ++k) {
              const int chunk = RotHalf<D>::channel(16 * k, p) / 16;  // of local values 16k..
              codes[(rw & 7) * kRowChunks + rot_code_chunk<D>(chunk, rw & 7)] = oc[k];
            }
          }
          __syncwarp();
          const int64_t row0 = tile * kRotTileRows + 16 * warp + 8 * h;
#pragma unroll
          for (int k = lane; k < kStageChunks; k += 32) {
            const int rr = k / kRowChunks, c = k - rr * kRowChunks;
            if (row0 + rr < rows)
              reinterpret_cast<uint4*>(x8 + (row0 + rr) * D)[c] =
                  codes[rr * kRowChunks + rot_code_chunk<D>(c, rr)];
          }
          __syncwarp();  // the next round's codes overwrite the buffer
        }
      }
    }
    if constexpr (!kQuant) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) warp_max[warp] = m;
    }
  }
  if constexpr (!kQuant) {
    __syncthreads();
    if (threadIdx.x == 0) {
      float r = 0.f;
      for (int i = 0; i < kRotConsumers; ++i) r = fmaxf(r, warp_max[i]);
      partial[blockIdx.x] = r;
    }
  }
}

template <int D, int XT>
int launch_rot_t(const CUtensorMap& tm, int64_t rows, const float* signs, void* x8,
                 float* descale, float* partial, int sms, cudaStream_t s) {
  using T = RotTile<D, XT>;
  auto k1 = rot_pass_kernel<D, XT, false>;
  auto k2 = rot_pass_kernel<D, XT, true>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
  if (e != cudaSuccess) return e;
  // Persistent grid: as many CTAs as are resident at once (both passes have
  // the same footprint), so that the static deal of tiles has no second wave.
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k2, kRotThreads, T::kSmem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t n_tiles = (rows + kRotTileRows - 1) / kRotTileRows;
  int cap = per_sm * sms;
  if (cap > kQuantMaxPartials) cap = kQuantMaxPartials;
  const int grid = n_tiles < 1 ? 1 : (n_tiles < cap ? static_cast<int>(n_tiles) : cap);
  k1<<<grid, kRotThreads, T::kSmem, s>>>(tm, rows, signs, partial, nullptr, nullptr, 0);
  k2<<<grid, kRotThreads, T::kSmem, s>>>(tm, rows, signs, partial, static_cast<uint8_t*>(x8),
                                         descale, grid);
  return cudaGetLastError();
}

}  // namespace

int launch_fp8_quantize(const void* x, int64_t n, int x_type, void* x8, float* descale,
                        float* partial, int sms, cudaStream_t stream) {
  if (x_type == kQuantBF16) return launch_t<kQuantBF16>(x, n, x8, descale, partial, sms, stream);
  if (x_type == kQuantF32) return launch_t<kQuantF32>(x, n, x8, descale, partial, sms, stream);
  return cudaErrorInvalidValue;
}

int launch_fp8_quantize_rotated(const CUtensorMap& tm, int64_t rows, int d, int x_type,
                                const float* signs, void* x8, float* descale, float* partial,
                                int sms, cudaStream_t stream) {
  if (d == 128 && x_type == kQuantBF16)
    return launch_rot_t<128, kQuantBF16>(tm, rows, signs, x8, descale, partial, sms, stream);
  if (d == 128 && x_type == kQuantF32)
    return launch_rot_t<128, kQuantF32>(tm, rows, signs, x8, descale, partial, sms, stream);
  if (d == 192 && x_type == kQuantBF16)
    return launch_rot_t<192, kQuantBF16>(tm, rows, signs, x8, descale, partial, sms, stream);
  if (d == 192 && x_type == kQuantF32)
    return launch_rot_t<192, kQuantF32>(tm, rows, signs, x8, descale, partial, sms, stream);
  return cudaErrorInvalidValue;
}

int rot_box_inner_elems(int x_type) { return x_type == kQuantBF16 ? 64 : 32; }

int read_rot_status(int* value, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_rot_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (reset) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_rot_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace zyfa

// ---------------------------------------------------------------------------
// Variant without a caller workspace, for callers that cannot allocate device
// memory: the per-CTA maxima of the first pass go to a file-scope array
// instead.  Every device that loads this library keeps these 4 KB until the
// process exits, and every call on a device shares them.
// ---------------------------------------------------------------------------
namespace zyfa {
namespace {

static __device__ __align__(256) float g_noalloc_partials[kQuantMaxPartials];
// The first pass launches at most kQuantMaxPartials CTAs (launch_t and
// launch_rot_t clamp their grids to it) and writes one maximum per CTA, so
// every input size fits the array.
static_assert(sizeof(g_noalloc_partials) / sizeof(float) >= kQuantMaxPartials,
              "the array holds one maximum per CTA of the largest first pass");

}  // namespace

int fp8_quantize_noalloc(const void* x, int64_t n, int x_type, void* x8, float* descale, int sms,
                         cudaStream_t stream) {
  // The array's device address is looked up on every call (a table lookup
  // once the module is loaded): a cached address would go stale when a
  // device reset reloads the module in a new context.
  void* partials = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&partials, g_noalloc_partials);
  if (e != cudaSuccess) return e;
  // Nothing needs clearing: the second pass reads only the slots the first
  // pass of the same call has written.
  return launch_fp8_quantize(x, n, x_type, x8, descale, static_cast<float*>(partials), sms,
                             stream);
}

}  // namespace zyfa
