// Single-feature GPU probe of the tensor-core encodings the attention kernel
// relies on, each checked against a CPU product in tests/test_gpu_probes.py:
//
//   mode 0 (SS): D[128x128] = A[128xK] * B[128xK]^T with A and B loaded by TMA
//                into 128-byte-swizzled K-major tiles (the S = Q K^T product);
//   mode 1 (TS): D[128x128] = A[128x128] * B[128x128] with A written into
//                tensor memory by tcgen05.st and B loaded by TMA as an MN-major
//                operand (the O += P V product);
//   mode 2/3 (TS, block-scaled, e4m3 only): as mode 1 with kind::mxf8f6f4 and
//                one UE8M0 scale per row of A per 32-deep slice of K (B's
//                scales all 2^0), the scale of row r and slice k written into
//                tensor memory at lane r, byte k of one column (mode 2), or
//                at lane 32q + r % 32 for every q, byte k of column r / 32
//                (mode 3).
//
// f8 selects kind::f8f6f4 with e4m3 operands instead of kind::f16 with BF16.
// One CTA of 128 threads; every wait is bounded.  A second probe lets a
// bounded wait run out (an arrival that never comes) and reports the status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "zyfa_ptx.cuh"

namespace {

using namespace zyfa;

__device__ int g_probe_status;

template <int F8, int MODE>
__global__ void __launch_bounds__(128, 1)
    mma_probe_kernel(const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b, const uint8_t* a_glob,
                     const uint8_t* sf_glob, float* d_out) {
  constexpr bool kBS = MODE >= 2;
  static_assert(!kBS || F8, "block scaling is an e4m3 form");
  constexpr int kElem = F8 ? 1 : 2;
  constexpr int kChunkElems = 128 / kElem;     // elements per 128-byte row chunk
  constexpr int kChunks = 128 * kElem / 128;   // chunks per 128-element row
  constexpr int kChunkBytes = 128 * 128;       // 128 rows x 128 bytes
  constexpr int kUmmaK = 32 / kElem;
  constexpr uint32_t kFmt = F8 ? 0u : 1u;
  constexpr uint32_t kIdesc = ptx::instr_desc(kFmt, kFmt, MODE >= 1 ? 1u : 0u, 128, 128);
  constexpr uint32_t kSfaCol = 192, kSfbCol = 224;   // scale factors of A and B

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sa = base;
  uint8_t* sb = base + kChunks * kChunkBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + kChunks * kChunkBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar_load = ptx::smem_u32(bars + 0);
  const uint32_t bar_mma = ptx::smem_u32(bars + 1);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_load, 1);
    ptx::mbar_init(bar_mma, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  __syncwarp();
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // D at columns [0,128), A (TS) at [128, ...), scale factors at 192 and 224.
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (threadIdx.x == 0) {
    const uint32_t bytes = (MODE == 0 ? 2 : 1) * kChunks * kChunkBytes;
    ptx::mbar_arrive_expect_tx(bar_load, bytes);
    for (int c = 0; c < kChunks; ++c) {
      if (MODE == 0)
        ptx::tma_load_4d_plain(ptx::smem_u32(sa + c * kChunkBytes), &tm_a, bar_load,
                               c * kChunkElems, 0, 0, 0);
      ptx::tma_load_4d_plain(ptx::smem_u32(sb + c * kChunkBytes), &tm_b, bar_load,
                             c * kChunkElems, 0, 0, 0);
    }
  }
  __syncwarp();
  if (MODE >= 1) {
    // Thread i writes row i of A (128 elements = 128*kElem bytes) into tensor
    // memory lane i, 4 bytes per column, in element order.
    const uint32_t* row = reinterpret_cast<const uint32_t*>(a_glob + threadIdx.x * 128 * kElem);
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int c = 0; c < 128 * kElem / 4; c += 32) {
      uint32_t r[32];
      for (int i = 0; i < 32; ++i) r[i] = row[c + i];
      ptx::tmem_st32(tmem + lane_base + 128 + c, r);
    }
    if constexpr (kBS) {
      const uint32_t ones[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
      ptx::tmem_st4(tmem + lane_base + kSfbCol, ones);
      auto word = [&](int r) {
        const uint8_t* e = sf_glob + r * 4;
        return uint32_t(e[0]) | (uint32_t(e[1]) << 8) | (uint32_t(e[2]) << 16) |
               (uint32_t(e[3]) << 24);
      };
      if (MODE == 2) {
        ptx::tmem_st1(tmem + lane_base + kSfaCol, word(threadIdx.x));
      } else if (MODE == 3) {
        const uint32_t w[4] = {word(lane), word(32 + lane), word(64 + lane), word(96 + lane)};
        ptx::tmem_st4(tmem + lane_base + kSfaCol, w);
      } else if (MODE == 4) {
        // own quadrant only: lane r, column r / 32; zeros elsewhere
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        w[warp] = word(threadIdx.x);
        ptx::tmem_st4(tmem + lane_base + kSfaCol, w);
      } else {
        // quadrant 0 only: lane r % 32, column r / 32; zeros elsewhere
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (warp == 0) {
          w[0] = word(lane); w[1] = word(32 + lane); w[2] = word(64 + lane); w[3] = word(96 + lane);
        }
        ptx::tmem_st4(tmem + lane_base + kSfaCol, w);
      }
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();

  if (threadIdx.x == 0) {
    ok = ptx::mbar_wait(bar_load, 0, abort_flag, &g_probe_status, 1);
    if (ok) {
      ptx::tc_fence_after();
      const uint32_t a_addr = ptx::smem_u32(sa), b_addr = ptx::smem_u32(sb);
      for (int ks = 0; ks < 128 / kUmmaK; ++ks) {
        if (MODE == 0) {
          const int c = ks * kUmmaK / kChunkElems;
          const int kk = (ks * kUmmaK % kChunkElems) * kElem;  // byte offset in the chunk row
          const uint32_t off = c * kChunkBytes + kk;
          ptx::mma_ss<F8>(tmem, ptx::smem_desc(a_addr + off, 16, 1024, 2u),
                          ptx::smem_desc(b_addr + off, 16, 1024, 2u), kIdesc, ks > 0);
        } else if constexpr (kBS) {
          // Slice ks takes byte ks of the scale-factor words.
          const uint32_t idesc = ptx::instr_desc_bs(0u, 0u, 1u, 128, 128, ks, ks);
          ptx::mma_ts_bs(tmem, tmem + 128 + ks * 8,
                         ptx::smem_desc(b_addr + ks * kUmmaK * 128, kChunkBytes, 1024, 2u),
                         idesc, tmem + kSfaCol, tmem + kSfbCol, ks > 0);
        } else {
          ptx::mma_ts<F8>(tmem, tmem + 128 + ks * 8,
                          ptx::smem_desc(b_addr + ks * kUmmaK * 128, kChunkBytes, 1024, 2u),
                          kIdesc, ks > 0);
        }
      }
      ptx::mma_commit(bar_mma);
      ok = ptx::mbar_wait(bar_mma, 0, abort_flag, &g_probe_status, 2);
      if (!ok) ptx::mbar_drain(bar_mma, 0);
    } else {
      ptx::mbar_drain(bar_load, 0);
    }
  }
  __syncwarp();
  __syncthreads();
  ptx::tc_fence_after();
  if (!*abort_flag) {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld32_wait(tmem + lane_base + c, r);
      for (int i = 0; i < 32; ++i) d_out[threadIdx.x * 128 + c + i] = __uint_as_float(r[i]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, 256);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A 128 x 128-element row-major matrix as a 4-D map (the last two dims 1),
// box = 128 rows x one 128-byte chunk, 128-byte swizzle.
int make_map(EncodeTiledFn enc, CUtensorMap* m, const void* p, int f8) {
  const cuuint64_t e = f8 ? 1 : 2;
  cuuint64_t dims[4] = {128, 128, 1, 1};
  cuuint64_t strides[3] = {128 * e, 128 * 128 * e, 128 * 128 * e};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / e), 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void*>(p), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int F8, int MODE>
int run(const CUtensorMap& a, const CUtensorMap& b, const void* a_glob, float* d,
        cudaStream_t s, const void* sf = nullptr) {
  auto k = mma_probe_kernel<F8, MODE>;
  const int smem = 1024 + 2 * 2 * 128 * 128 + 256;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<1, 128, smem, s>>>(a, b, static_cast<const uint8_t*>(a_glob),
                         static_cast<const uint8_t*>(sf), d);
  return cudaGetLastError();
}

// Wait-timeout probe: one thread waits on an mbarrier that nothing ever
// arrives at, with the attention kernel's bounded wait.  out[0] = 1 when the
// wait (wrongly) reported success, out[1] = the abort flag it raised, out[2]
// = elapsed global time in microseconds.  The failure is made by withholding
// the arrival; nothing faults and the wait ends by itself.
__global__ void wait_timeout_probe_kernel(int* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer();
    const bool ok = ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, &g_probe_status, 1);
    out[0] = ok ? 1 : 0;
    out[1] = abort_flag;
    out[2] = static_cast<int>((ptx::globaltimer() - t0) / 1000);
  }
}

}  // namespace

extern "C" {

// Runs wait_timeout_probe_kernel (one thread; about kWaitTimeoutNs of wall
// time) and synchronises; out: device, 3 ints.  Returns a cudaError_t.
__attribute__((visibility("default"))) int zyfa_probe_wait_timeout(int* out) {
  wait_timeout_probe_kernel<<<1, 32>>>(out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return cudaDeviceSynchronize();
}

__attribute__((visibility("default"))) int zyfa_probe_status_reset(void) {
  const int zero = 0;
  return cudaMemcpyToSymbol(g_probe_status, &zero, sizeof(int));
}


// a, b: device 128x128 row-major (BF16 or e4m3 codes); d: device FP32 128x128.
// mode 0: d = a * b^T (both K-major, SS); mode 1: d = a * b (a via TMEM, b MN-major).
__attribute__((visibility("default"))) int zyfa_probe_mma(int f8, int mode, const void* a, const void* b, float* d, void* stream) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return -5;
  auto enc = reinterpret_cast<EncodeTiledFn>(fn);
  CUtensorMap ma, mb;
  if (make_map(enc, &ma, a, f8) != CUDA_SUCCESS || make_map(enc, &mb, b, f8) != CUDA_SUCCESS)
    return -1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (f8 == 0 && mode == 0) return run<0, 0>(ma, mb, a, d, s);
  if (f8 == 0 && mode == 1) return run<0, 1>(ma, mb, a, d, s);
  if (f8 == 1 && mode == 0) return run<1, 0>(ma, mb, a, d, s);
  if (f8 == 1 && mode == 1) return run<1, 1>(ma, mb, a, d, s);
  return -1;
}

// Block-scaled form: a, b as mode 1 (e4m3 codes), sf: device 128 x 4 bytes,
// the UE8M0 scale of row r of a and K slice k at sf[4 r + k]; layout 0
// writes them as mode 2 of the probe kernel, layout 1 as mode 3.
// d = (a x 2^(sf - 127)) * b.
__attribute__((visibility("default"))) int zyfa_probe_mma_bs(int layout, const void* a, const void* b,
                                                             const void* sf, float* d, void* stream) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return -5;
  auto enc = reinterpret_cast<EncodeTiledFn>(fn);
  CUtensorMap ma, mb;
  if (make_map(enc, &ma, a, 1) != CUDA_SUCCESS || make_map(enc, &mb, b, 1) != CUDA_SUCCESS)
    return -1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (layout == 0) return run<1, 2>(ma, mb, a, d, s, sf);
  if (layout == 1) return run<1, 3>(ma, mb, a, d, s, sf);
  if (layout == 2) return run<1, 4>(ma, mb, a, d, s, sf);
  if (layout == 3) return run<1, 5>(ma, mb, a, d, s, sf);
  return -1;
}

__attribute__((visibility("default"))) int zyfa_probe_status(int* v) {
  return cudaMemcpyFromSymbol(v, g_probe_status, sizeof(int));
}

}  // extern "C"
