// Internal interface of the FP8 quantisation kernels (quant.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace zyfa {

constexpr int kQuantBF16 = 0;          // input element types (ZYFA_BF16, ZYFA_F32)
constexpr int kQuantF32 = 2;
constexpr int kQuantMaxPartials = 1024; // CTAs of the max pass = floats of workspace

// Enqueues the two quantisation passes; `partial` holds kQuantMaxPartials
// floats.  Returns a cudaError_t.
int launch_fp8_quantize(const void* x, int64_t n, int x_type, void* x8, float* descale,
                        float* partial, int sms, cudaStream_t stream);

// Rows of d = 128 or 192 channels rotated by diag(signs) times the Hadamard
// (d = 128) or DCT x Hadamard (d = 192) matrix, then quantised per tensor like
// launch_fp8_quantize.  `tm` is a 2-D tensor map over x as (d channels, rows)
// with a box of 64 rows x rot_box_inner_elems(x_type) channels (128 bytes)
// and 128-byte swizzle.  Returns a cudaError_t.
int launch_fp8_quantize_rotated(const CUtensorMap& tm, int64_t rows, int d, int x_type,
                                const float* signs, void* x8, float* descale, float* partial,
                                int sms, cudaStream_t stream);
int rot_box_inner_elems(int x_type);
constexpr int kRotBoxRows = 64;

// Status word of the rotation kernels (bit 0: a wait timed out).
int read_rot_status(int* value, int reset);

// Same, with the first pass's maxima in a file-scope device array instead of a
// caller workspace (one-time symbol lookup per device on first use).
int fp8_quantize_noalloc(const void* x, int64_t n, int x_type, void* x8, float* descale, int sms,
                         cudaStream_t stream);

}  // namespace zyfa
