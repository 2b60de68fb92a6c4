// Internal interface between the C-ABI layer (api.cpp) and the kernel
// translation unit (fwd_sm103.cu).  Not part of the public header.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace zyfa {

// Everything one launch needs besides the three tensor maps.
struct FwdParams {
  void* out;                 // BF16 O, caller's layout
  float* lse;                // FP32 (B, H, S) or nullptr
  const float* q_descale;    // device scalars (FP8 only, else nullptr)
  const float* k_descale;
  const float* v_descale;
  int B, S, H, Hkv;
  int layout;                // 0 = bshd, 1 = bhsd
  int n_qblocks;             // ceil(S / 256): query blocks of two 128-row tiles
  int total_items;           // B * H * n_qblocks
  int serialize_pv;          // verification mode: P fully read before S reuses it
  int rounded_p;             // 0: default; 1: O's denominator from the rounded P on
                             // every tile; 2: that and the LSE from the same sum
  int block_scale;           // FP8: P scaled per 32-key slice, block-scaled P V
  int dynamic_schedule;      // one CTA per item, items taken by cancelling CTAs
  float softmax_scale;
};

struct TensorMaps {
  CUtensorMap q, k, v;
};

// Launches the forward kernel for (dtype, d_qk) on the current device, whose
// index (below 64) is `device`.  Returns a cudaError_t.
int launch_fwd(int dtype, int d_qk, const FwdParams& p, const TensorMaps& maps, int grid,
               int device, cudaStream_t stream);

// Dynamic shared memory bytes and swizzle geometry of an instantiation, so the
// host builds tensor maps whose boxes match the kernel's shared-memory tiles.
struct KernelGeometry {
  int smem_bytes;
  int qk_box_elems;    // inner box extent (elements) of Q and K loads
  int qk_swizzle;      // 128 or 64 (bytes)
  int v_box_elems;     // inner box extent of V loads (128-byte swizzle)
  int num_slots;       // K/V ring entries (whole-tile slots or 16 KB pieces)
};
int kernel_geometry(int dtype, int d_qk, KernelGeometry* g);

// Device-side status word (bit 0: a wait timed out).
int read_device_status(int* value, int reset);

}  // namespace zyfa
