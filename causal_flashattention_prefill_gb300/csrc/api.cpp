// C ABI of the causal prefill attention library: argument validation, TMA
// tensor-map encoding for the bshd/bhsd layouts, and the launch.  See
// include/zyfa.h for the contract of every entry point.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fwd.h"
#include "quant.h"
#include "zyfa.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::atomic<int> g_serialize_pv{0};
std::atomic<int> g_rounded_p{0};
std::atomic<int> g_block_scale{0};
std::atomic<int> g_dynamic_schedule{0};

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int checked = 0;  // 0 = not yet, 1 = usable, -1 = unusable
  int sm_count = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
bool g_encode_checked = false;

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_checked) {
    g_encode_checked = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// Returns the SM count of the current device, or -1 when it is not an
// sm_103 device; *device_out (optional) receives the device index.
int current_device_sms(int* device_out = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  if (device_out) *device_out = dev;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    d.checked = (major == 10 && minor == 3 && sms > 0) ? 1 : -1;
    d.sm_count = sms;
  }
  return d.checked == 1 ? d.sm_count : -1;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tensor maps of recent calls, keyed by everything they encode (base
// addresses, sizes, layout, element type; the box geometry follows from
// dtype and d_qk).  A map holds no device state, so an entry stays valid
// whatever happens to the buffers; repeated calls on the same buffers skip
// the three encodings.
struct MapKey {
  const void* q;
  const void* k;
  const void* v;
  int dtype, layout, B, S, H, Hkv, d_qk, d_v;
  bool operator==(const MapKey& o) const {
    return q == o.q && k == o.k && v == o.v && dtype == o.dtype && layout == o.layout &&
           B == o.B && S == o.S && H == o.H && Hkv == o.Hkv && d_qk == o.d_qk && d_v == o.d_v;
  }
};
struct MapEntry {
  MapKey key;
  zyfa::TensorMaps maps;
  bool valid = false;
};
constexpr int kMapCacheEntries = 16;
MapEntry g_map_cache[kMapCacheEntries];
int g_map_cache_next = 0;

bool cached_maps(const MapKey& key, zyfa::TensorMaps* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (const MapEntry& e : g_map_cache) {
    if (e.valid && e.key == key) {
      *out = e.maps;
      return true;
    }
  }
  return false;
}

void remember_maps(const MapKey& key, const zyfa::TensorMaps& maps) {
  std::lock_guard<std::mutex> lk(g_mu);
  MapEntry& e = g_map_cache[g_map_cache_next];
  g_map_cache_next = (g_map_cache_next + 1) % kMapCacheEntries;
  e.key = key;
  e.maps = maps;
  e.valid = true;
}

int validate(const void* q, const void* k, const void* v, void* out, float* lse, int B, int S,
             int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
             const float* k_descale, const float* v_descale, float scale, int layout) {
  if (!q || !k || !v || !out) return ZYFA_ERR_ARG;
  if (B < 1 || S < 1 || H < 1 || Hkv < 1) return ZYFA_ERR_ARG;
  if (H % Hkv != 0) return ZYFA_ERR_ARG;
  if (layout != ZYFA_BSHD && layout != ZYFA_BHSD) return ZYFA_ERR_ARG;
  if (d_qk < 1 || d_v < 1) return ZYFA_ERR_ARG;
  if (!((d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128))) return ZYFA_ERR_UNSUPPORTED;
  if (dtype != ZYFA_BF16 && dtype != ZYFA_FP8_E4M3) return ZYFA_ERR_UNSUPPORTED;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return ZYFA_ERR_ARG;
  if (dtype == ZYFA_FP8_E4M3) {
    if (!q_descale || !k_descale || !v_descale) return ZYFA_ERR_ARG;
    if (!aligned(q_descale, 4) || !aligned(k_descale, 4) || !aligned(v_descale, 4))
      return ZYFA_ERR_ALIGN;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return ZYFA_ERR_ALIGN;
  if (lse && !aligned(lse, 4)) return ZYFA_ERR_ALIGN;
  // Index ranges: work items and TMA coordinates are 32-bit, byte strides of
  // a tensor map must stay below 2^40.
  const int64_t n_qblocks = (static_cast<int64_t>(S) + 255) / 256;
  if (static_cast<int64_t>(B) * H * n_qblocks > INT_MAX) return ZYFA_ERR_UNSUPPORTED;
  const int64_t e = dtype == ZYFA_BF16 ? 2 : 1;
  const int64_t batch_stride_bytes = static_cast<int64_t>(S) * H * d_qk * e;  // largest stride
  if (batch_stride_bytes >= (int64_t(1) << 40)) return ZYFA_ERR_UNSUPPORTED;
  return ZYFA_OK;
}

// 4-D map over (d, heads, S, B) for bshd or (d, S, heads, B) for bhsd; the
// box is 128 sequence rows of `box_inner` elements of one head, with
// `swizzle` bytes of swizzle.
int make_map(CUtensorMap* m, const void* base, int dtype, int layout, int B, int S, int heads,
             int d, int box_inner, int swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return ZYFA_ERR_DEVICE;
  const cuuint64_t e = dtype == ZYFA_BF16 ? 2 : 1;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (layout == ZYFA_BSHD) {
    dims[0] = d; dims[1] = heads; dims[2] = S; dims[3] = B;
    strides[0] = d * e;
    strides[1] = static_cast<cuuint64_t>(heads) * d * e;
    strides[2] = static_cast<cuuint64_t>(S) * heads * d * e;
    box[0] = box_inner; box[1] = 1; box[2] = 128; box[3] = 1;
  } else {
    dims[0] = d; dims[1] = S; dims[2] = heads; dims[3] = B;
    strides[0] = d * e;
    strides[1] = static_cast<cuuint64_t>(S) * d * e;
    strides[2] = static_cast<cuuint64_t>(heads) * S * d * e;
    box[0] = box_inner; box[1] = 128; box[2] = 1; box[3] = 1;
  }
  const CUtensorMapDataType dt =
      dtype == ZYFA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle sw =
      swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ZYFA_OK : ZYFA_ERR_ARG;
}

// 2-D map over rows of d channels (x_type elements, rows contiguous): box of
// 64 rows x 128 bytes, 128-byte swizzle (the rotation kernels' tiles).  An
// empty tensor still gets a valid map (one row); no copy is issued then.
int make_rows_map(CUtensorMap* m, const void* base, int x_type, long long rows, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return ZYFA_ERR_DEVICE;
  const cuuint64_t e = x_type == zyfa::kQuantBF16 ? 2 : 4;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d),
                              static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * e};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(zyfa::rot_box_inner_elems(x_type)),
                             static_cast<cuuint32_t>(zyfa::kRotBoxRows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = x_type == zyfa::kQuantBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ZYFA_OK : ZYFA_ERR_ARG;
}

}  // namespace

extern "C" {

int zyfa_validate(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                  int S, int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
                  const float* k_descale, const float* v_descale, float softmax_scale,
                  int layout) {
  return validate(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale, k_descale,
                  v_descale, softmax_scale, layout);
}

int zyfa_fwd_scaled(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int S, int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
                    const float* k_descale, const float* v_descale, float softmax_scale,
                    int layout, struct CUstream_st* stream) {
  int st = validate(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale, k_descale,
                    v_descale, softmax_scale, layout);
  if (st != ZYFA_OK) return st;
  int device = 0;
  const int sms = current_device_sms(&device);
  if (sms <= 0) return ZYFA_ERR_DEVICE;

  zyfa::KernelGeometry g;
  if (zyfa::kernel_geometry(dtype, d_qk, &g) != 0) return ZYFA_ERR_UNSUPPORTED;
  zyfa::TensorMaps maps;
  const MapKey key{q, k, v, dtype, layout, B, S, H, Hkv, d_qk, d_v};
  if (!cached_maps(key, &maps)) {
    std::memset(&maps, 0, sizeof(maps));
    if ((st = make_map(&maps.q, q, dtype, layout, B, S, H, d_qk, g.qk_box_elems, g.qk_swizzle)))
      return st;
    if ((st = make_map(&maps.k, k, dtype, layout, B, S, Hkv, d_qk, g.qk_box_elems, g.qk_swizzle)))
      return st;
    if ((st = make_map(&maps.v, v, dtype, layout, B, S, Hkv, d_v, g.v_box_elems, 128))) return st;
    remember_maps(key, maps);
  }

  zyfa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.out = out;
  p.lse = lse;
  if (dtype == ZYFA_FP8_E4M3) {
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
  }
  p.B = B;
  p.S = S;
  p.H = H;
  p.Hkv = Hkv;
  p.layout = layout;
  p.n_qblocks = (S + 255) / 256;
  p.total_items = B * H * p.n_qblocks;
  p.serialize_pv = g_serialize_pv.load(std::memory_order_relaxed);
  p.rounded_p = g_rounded_p.load(std::memory_order_relaxed);
  p.block_scale = g_block_scale.load(std::memory_order_relaxed);
  p.dynamic_schedule = g_dynamic_schedule.load(std::memory_order_relaxed);
  p.softmax_scale = softmax_scale;
  // Static schedule: one persistent CTA per SM.  Dynamic: one CTA per item,
  // of which about one per SM runs at a time and takes the items of the
  // CTAs that have not started.
  // (The dynamic schedule covers the default softmax modes; with the
  // rounded-P or block-scaled options the static one is used.)
  if (p.rounded_p != 0 || (dtype == ZYFA_FP8_E4M3 && p.block_scale != 0)) p.dynamic_schedule = 0;
  const int grid = (p.dynamic_schedule || p.total_items < sms) ? p.total_items : sms;
  const int e = zyfa::launch_fwd(dtype, d_qk, p, maps, grid, device,
                                 reinterpret_cast<cudaStream_t>(stream));
  return e == 0 ? ZYFA_OK : ZYFA_ERR_LAUNCH;
}

int zyfa_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int S,
             int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
             const float* k_descale, const float* v_descale, int layout,
             struct CUstream_st* stream) {
  const float scale = d_qk > 0 ? 1.0f / std::sqrt(static_cast<float>(d_qk)) : 0.0f;
  return zyfa_fwd_scaled(q, k, v, out, lse, B, S, H, Hkv, d_qk, d_v, dtype, q_descale, k_descale,
                         v_descale, scale, layout, stream);
}

const char* zyfa_status_string(int status) {
  switch (status) {
    case ZYFA_OK: return "ok";
    case ZYFA_ERR_ARG: return "invalid argument";
    case ZYFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case ZYFA_ERR_ALIGN: return "misaligned pointer";
    case ZYFA_ERR_LAUNCH: return "kernel launch failed";
    case ZYFA_ERR_DEVICE: return "no usable sm_103 device or driver entry point";
    case ZYFA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    default: return "unknown status";
  }
}

int zyfa_device_status(int* value, int reset) {
  if (!value) return ZYFA_ERR_ARG;
  // The attention kernel and the rotation kernels keep separate words (one
  // per translation unit); the reported word is their union.
  int a = 0, r = 0;
  if (zyfa::read_device_status(&a, reset) != 0) return ZYFA_ERR_DEVICE;
  if (zyfa::read_rot_status(&r, reset) != 0) return ZYFA_ERR_DEVICE;
  *value = a | r;
  return ZYFA_OK;
}

int zyfa_set_option(int option, int value) {
  if (option == ZYFA_OPT_SERIALIZE_PV) {
    g_serialize_pv.store(value ? 1 : 0);
    return ZYFA_OK;
  }
  if (option == ZYFA_OPT_ROUNDED_P) {
    if (value < 0 || value > 2) return ZYFA_ERR_ARG;
    g_rounded_p.store(value);
    return ZYFA_OK;
  }
  if (option == ZYFA_OPT_BLOCK_SCALE) {
    if (value < 0 || value > 1) return ZYFA_ERR_ARG;
    g_block_scale.store(value);
    return ZYFA_OK;
  }
  if (option == ZYFA_OPT_DYNAMIC_SCHEDULE) {
    if (value < 0 || value > 1) return ZYFA_ERR_ARG;
    g_dynamic_schedule.store(value);
    return ZYFA_OK;
  }
  return ZYFA_ERR_ARG;
}

long long zyfa_fp8_quantize_workspace_bytes(void) {
  return static_cast<long long>(zyfa::kQuantMaxPartials) * sizeof(float);
}

int zyfa_fp8_quantize(const void* x, long long n, int x_dtype, void* x8, float* descale,
                      void* workspace, struct CUstream_st* stream) {
  if (!x || !x8 || !descale || !workspace || n < 0) return ZYFA_ERR_ARG;
  if (x_dtype != ZYFA_BF16 && x_dtype != ZYFA_F32) return ZYFA_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(x8, 8) || !aligned(descale, 4) || !aligned(workspace, 4))
    return ZYFA_ERR_ALIGN;
  const int sms = current_device_sms();
  if (sms <= 0) return ZYFA_ERR_DEVICE;
  const int e = zyfa::launch_fp8_quantize(x, n, x_dtype == ZYFA_BF16 ? zyfa::kQuantBF16
                                                                      : zyfa::kQuantF32,
                                          x8, descale, static_cast<float*>(workspace), sms,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == 0 ? ZYFA_OK : ZYFA_ERR_LAUNCH;
}

int zyfa_fp8_quantize_noalloc(const void* x, long long n, int x_dtype, void* x8,
                              float* descale, struct CUstream_st* stream) {
  if (!x || !x8 || !descale || n < 0) return ZYFA_ERR_ARG;
  if (x_dtype != ZYFA_BF16 && x_dtype != ZYFA_F32) return ZYFA_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(x8, 8) || !aligned(descale, 4)) return ZYFA_ERR_ALIGN;
  const int sms = current_device_sms();
  if (sms <= 0) return ZYFA_ERR_DEVICE;
  const int e = zyfa::fp8_quantize_noalloc(
      x, n, x_dtype == ZYFA_BF16 ? zyfa::kQuantBF16 : zyfa::kQuantF32, x8, descale, sms,
      reinterpret_cast<cudaStream_t>(stream));
  return e == 0 ? ZYFA_OK : ZYFA_ERR_LAUNCH;
}

int zyfa_fp8_quantize_rotated(const void* x, long long n_rows, int d, int x_dtype,
                              const float* signs, void* x8, float* descale, void* workspace,
                              struct CUstream_st* stream) {
  if (!x || !signs || !x8 || !descale || !workspace || n_rows < 0) return ZYFA_ERR_ARG;
  if (d != 128 && d != 192) return ZYFA_ERR_UNSUPPORTED;
  if (x_dtype != ZYFA_BF16 && x_dtype != ZYFA_F32) return ZYFA_ERR_UNSUPPORTED;
  if (n_rows > (1LL << 40) / d) return ZYFA_ERR_ARG;
  // Tile coordinates of the copies are 32-bit row indices.
  if (n_rows > (1LL << 31) - 1 - zyfa::kRotBoxRows) return ZYFA_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(descale, 4) || !aligned(workspace, 4) ||
      !aligned(signs, 4))
    return ZYFA_ERR_ALIGN;
  const int sms = current_device_sms();
  if (sms <= 0) return ZYFA_ERR_DEVICE;
  const int xt = x_dtype == ZYFA_BF16 ? zyfa::kQuantBF16 : zyfa::kQuantF32;
  CUtensorMap tm;
  const int me = make_rows_map(&tm, x, xt, n_rows, d);
  if (me != ZYFA_OK) return me;
  const int e = zyfa::launch_fp8_quantize_rotated(tm, n_rows, d, xt, signs, x8, descale,
                                                  static_cast<float*>(workspace), sms,
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == 0 ? ZYFA_OK : ZYFA_ERR_LAUNCH;
}

int zyfa_version(void) { return (1 << 16) | 1; }

}  // extern "C"
