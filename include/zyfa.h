/*
 * zyfa.h -- C ABI of the GB300 (sm_103a) causal prefill attention library.
 *
 * The operation is the causal forward attention pass for inference prefill
 * that the ZYFA README defines ("Usage" and "Supported configurations"):
 *
 *   O[b, i, h, :] = sum_{j <= i} softmax_j(scale * <q[b,i,h], k[b,j,hk]>) v[b,j,hk]
 *   LSE[b, h, i]  = ln sum_{j <= i} exp(scale * <q[b,i,h], k[b,j,hk]>)
 *
 * with seqlen_q = seqlen_k = S, equal-length batches, hk = h / (H / Hkv)
 * (MHA, GQA and MQA: the query-head count is any multiple of the KV-head
 * count), head dims d_qk = d_v = 128 or d_qk = 192 with d_v = 128, BF16 or
 * FP8 e4m3 inputs with one descale per tensor (the kernel itself loads the
 * three descales from device memory and applies them, so no call waits for
 * the host; "Usage"), BF16 output and an optional FP32 natural-log LSE of the
 * scaled scores.  Any S >= 1 is accepted: lengths that are not a multiple of the tile
 * give the same result as zero-padding ("Usage": padding is exact for causal
 * attention), with no copy.
 *
 * Layouts (all tensors dense and contiguous, element strides implied):
 *   ZYFA_BSHD: q (B,S,H,d_qk)  k (B,S,Hkv,d_qk)  v (B,S,Hkv,d_v)  out (B,S,H,d_v)
 *   ZYFA_BHSD: q (B,H,S,d_qk)  k (B,Hkv,S,d_qk)  v (B,Hkv,S,d_v)  out (B,H,S,d_v)
 *   lse is (B,H,S) FP32 in both layouts.
 *
 * Ownership and synchronisation: every pointer is a device pointer owned by
 * the caller.  The library allocates nothing per call (no workspace, no host
 * job table) and never synchronises the host: a call only enqueues one kernel
 * on `stream`, so it can be captured in a CUDA graph from the first call.
 *
 * Errors: argument checks run on the host before any CUDA call and return a
 * negative zyfa_status without launching anything.  Launch failures return
 * ZYFA_ERR_LAUNCH.  Asynchronous device errors surface on the caller's next
 * synchronisation.  Every wait inside the kernel is bounded (2 s); a wait that
 * runs out makes the kernel unwind and sets bit 0 of the device status word
 * read by zyfa_device_status().
 */
#ifndef ZYFA_H
#define ZYFA_H

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ZYFA_API __attribute__((visibility("default")))
#else
#define ZYFA_API
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st*`; NULL = default stream */

typedef enum {
  ZYFA_OK = 0,
  ZYFA_ERR_ARG = -1,            /* invalid value (sizes, enums, NULL pointers)       */
  ZYFA_ERR_UNSUPPORTED = -2,    /* valid request outside the supported configurations */
  ZYFA_ERR_ALIGN = -3,          /* a pointer is not 16-byte aligned (lse: 4-byte)   */
  ZYFA_ERR_LAUNCH = -4,         /* the kernel launch failed                          */
  ZYFA_ERR_DEVICE = -5,         /* no usable sm_103 device / driver entry point      */
  ZYFA_ERR_DEVICE_TIMEOUT = -6  /* reported by zyfa_device_status()                  */
} zyfa_status;

enum { ZYFA_BF16 = 0, ZYFA_FP8_E4M3 = 1, ZYFA_F32 = 2 };
enum { ZYFA_BSHD = 0, ZYFA_BHSD = 1 };

/*
 * Causal forward attention with softmax_scale = 1/sqrt(d_qk).
 *
 * q, k, v    device, BF16 (dtype ZYFA_BF16) or e4m3 codes (ZYFA_FP8_E4M3),
 *            16-byte aligned, shapes per `layout` above.
 * out        device, BF16, 16-byte aligned; written for every (b, i, h).
 * lse        device FP32 (B,H,S), 4-byte aligned, or NULL to skip it.
 * B, S       batch size >= 1 and sequence length >= 1 (queries = keys = S).
 * H, Hkv     query heads and KV heads, H % Hkv == 0.
 * d_qk, d_v  (128, 128) or (192, 128).
 * q_descale, k_descale, v_descale
 *            FP8: device pointers to one FP32 each (the factor that maps
 *            the e4m3 tensor back to its range); the values must be positive
 *            normal floats and are not checked.  BF16: ignored (may be NULL).
 * layout     ZYFA_BSHD or ZYFA_BHSD.
 * stream     CUDA stream the kernel is enqueued on.
 * Returns ZYFA_OK or a negative zyfa_status.
 */
ZYFA_API int zyfa_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int S,
             int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
             const float* k_descale, const float* v_descale, int layout,
             struct CUstream_st* stream);

/*
 * zyfa_fwd with an explicit softmax_scale (finite, > 0): the scale argument of
 * flash_attn_func in the ZYFA README ("Usage"; "Differences from flash-attn":
 * the flash-attn calling convention, scale default 1/sqrt(head dim)).  The
 * scale multiplies the scores before the softmax and enters the LSE; for FP8
 * inputs it is applied on top of q_descale * k_descale.  Other arguments,
 * ownership and errors as zyfa_fwd (a scale that is not finite and positive
 * returns ZYFA_ERR_ARG before any CUDA call).
 */
ZYFA_API int zyfa_fwd_scaled(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                    int S, int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
                    const float* k_descale, const float* v_descale, float softmax_scale,
                    int layout, struct CUstream_st* stream);

/*
 * Runs only the host-side argument checks of zyfa_fwd_scaled, with no CUDA
 * call (the supported configurations of the ZYFA README, "Supported
 * configurations": causal, seqlen_q = seqlen_k, head dims (128, 128) or
 * (192, 128), query heads a multiple of KV heads, BF16 or FP8 e4m3 inputs;
 * "Usage": FP8 needs all three descales).  Pointers are only checked for
 * NULL and alignment, never dereferenced.  Returns ZYFA_OK when
 * zyfa_fwd_scaled would launch, else the status that call would return.
 */
ZYFA_API int zyfa_validate(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                  int S, int H, int Hkv, int d_qk, int d_v, int dtype, const float* q_descale,
                  const float* k_descale, const float* v_descale, float softmax_scale,
                  int layout);

/*
 * Static English description of a zyfa_status value (unknown values give
 * "unknown status"); never NULL, owned by the library.  The statuses are how
 * this C interface reports the rejections the ZYFA README lists under
 * "Supported configurations" (ZYFA_ERR_UNSUPPORTED) and invalid arguments.
 */
ZYFA_API const char* zyfa_status_string(int status);

/*
 * Reads the device status word of the current device into *value (0 = no
 * wait has timed out; bit 0 = a wait of the attention kernel or of the
 * rotation kernels timed out) and clears it when `reset` is non-zero.
 * Synchronous.  Returns ZYFA_OK or ZYFA_ERR_DEVICE.
 */
ZYFA_API int zyfa_device_status(int* value, int reset);

/*
 * Library options (process-wide; take effect on the next call).
 *   ZYFA_OPT_SERIALIZE_PV: when 1, the kernel waits for each P*V product to
 *   finish before the next score product of the same query tile overwrites
 *   the tensor memory that holds P.  Results are identical; it exists to
 *   verify that the default pipelined order is race-free.  Default 0.
 *   ZYFA_OPT_ROUNDED_P: how the sums of the probabilities are formed (the
 *   ZYFA README, "Accuracy" and "Kernel design": the output is divided by
 *   the sum of the same rounded probabilities that multiply V, and the FP8
 *   log-sum-exp comes from the rounded probabilities so that results over
 *   different key ranges merge consistently).
 *     0 (default): the denominator is the sum of the rounded P (the BF16
 *       values, or for FP8 the two e4m3 terms) on tiles where one
 *       probability carries a large share of the row's mass, the unrounded
 *       sum elsewhere; the LSE comes from the unrounded sum.
 *     1: the denominator is the sum of the rounded P that multiplies V on
 *       every tile, so each output row is a weighted average whose weights
 *       sum to one; the LSE as in 0.
 *     2: as 1, and the LSE is taken from that same rounded sum.
 *   Modes 1 and 2 add work to every tile of the softmax (slower).
 *   ZYFA_OPT_BLOCK_SCALE (FP8 calls; BF16 calls ignore it): when 1, P is
 *   scaled per row and 32-key slice by the power of two that brings the
 *   slice's largest probability into the binade of p = 1 before it is
 *   rounded to e4m3, and the P*V product is the block-scaled MMA, which
 *   divides the same power of two back out (ZYFA README, "Kernel design":
 *   per-block scaling, which keeps probabilities far below the row maximum
 *   normal instead of subnormal or zero; GB300's scale blocks are 32 keys,
 *   the page's 64).  Combines with ZYFA_OPT_ROUNDED_P.  Default 0; slower.
 *   ZYFA_OPT_DYNAMIC_SCHEDULE: when 1, work items (query blocks of 256 rows
 *   of one head) go to whichever SM frees up first, longest first, instead
 *   of the static deal over one persistent CTA per SM (ZYFA README, "Kernel
 *   design": longest-first work distribution).  The outputs are the same
 *   bits either way; dynamic helps when the cost of an item varies with the
 *   data (rows whose maximum keeps rising), static is slightly faster on
 *   regular rows.  It applies to the default softmax modes: with
 *   ZYFA_OPT_ROUNDED_P or (FP8) ZYFA_OPT_BLOCK_SCALE set, the static
 *   schedule is used.  Default 0.
 * Returns ZYFA_OK or ZYFA_ERR_ARG.
 */
enum {
  ZYFA_OPT_SERIALIZE_PV = 1,
  ZYFA_OPT_ROUNDED_P = 2,
  ZYFA_OPT_BLOCK_SCALE = 3,
  ZYFA_OPT_DYNAMIC_SCHEDULE = 4
};
ZYFA_API int zyfa_set_option(int option, int value);

/*
 * Per-tensor FP8 quantisation (the input preparation of the FP8 path; ZYFA
 * README, "Usage": fp8_quantize returns the e4m3 tensor and one power-of-two
 * descale per tensor as a GPU scalar; "Kernel design": all conversions use
 * round-half-to-even).
 *
 *   descale = smallest power of two with max|x| / descale <= 448 (1 if x is
 *             all zero);   x8[i] = e4m3(x[i] / descale), ties to even,
 *             saturating to +-448.
 *
 * x          device, n elements of x_dtype (ZYFA_BF16 or ZYFA_F32), 16-byte
 *            aligned; NaN inputs give unspecified results.
 * n          element count (>= 0).
 * x8         device, n bytes of e4m3 codes, 8-byte aligned.
 * descale    device, one FP32, written by the kernel (the host never waits).
 * workspace  device scratch of zyfa_fp8_quantize_workspace_bytes() bytes,
 *            4-byte aligned, owned by the caller; its contents need no
 *            initialisation and are meaningless after the call.  Calls that
 *            may overlap on the GPU need separate workspaces.
 * Two kernels are enqueued on `stream`; deterministic (no atomics).
 * Returns ZYFA_OK or a negative zyfa_status (checks run before any launch).
 */
ZYFA_API int zyfa_fp8_quantize(const void* x, long long n, int x_dtype, void* x8, float* descale,
                               void* workspace, struct CUstream_st* stream);

/* Bytes of workspace zyfa_fp8_quantize needs (a constant). */
ZYFA_API long long zyfa_fp8_quantize_workspace_bytes(void);

/*
 * zyfa_fp8_quantize without a workspace argument, for callers that cannot
 * allocate device memory: code that only receives the buffers a host
 * framework planned for it (a fixed memory arena, a plugin interface that
 * hands over inputs and outputs only), or that runs where an allocation
 * would stall the device.  The pages have no counterpart to this entry
 * point; it is a deployment convenience.
 *
 * Same arguments, results and errors as zyfa_fp8_quantize, minus
 * `workspace`.  The scratch it needs (one FP32 maximum per CTA of the first
 * pass, at most 1024 of them) lives in a 4 KB array inside this library,
 * kept on every device that runs this entry point until the process exits.
 * The first pass never launches more CTAs than the array has slots, so every
 * input size fits.  Nothing in the array has to start at zero, but all calls
 * on a device share it, so calls that may run at the same time on the GPU
 * (on different streams without ordering) race and must not be made.  The
 * first call on each device looks up the array's device address (a CUDA
 * runtime call) and should come before any stream capture; the address is
 * kept for the life of the process, so after cudaDeviceReset on a device
 * this entry point must not be called on that device again.  The entry
 * point never allocates: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 */
ZYFA_API int zyfa_fp8_quantize_noalloc(const void* x, long long n, int x_dtype, void* x8,
                                       float* descale, struct CUstream_st* stream);

/*
 * Rotation of q or k followed by per-tensor FP8 quantisation, in two kernels
 * (ZYFA README, "Using FP8 attention in a model": a Hadamard rotation of q
 * and k before quantisation roughly halves the input error, and fused into
 * the pass that quantises q it costs little; v is left unrotated).  Each row
 * of d channels is rotated as y = x @ R with
 *
 *   d = 128: R = diag(signs) H / sqrt(128), H Sylvester's Hadamard matrix
 *            (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]);
 *   d = 192: R = diag(signs) (C3^T kron H_64) / 8, C3 the orthonormal 3-point
 *            DCT-II (C3[k][n] = a_k cos(pi (2n+1) k / 6), a_0 = sqrt(1/3),
 *            a_k = sqrt(2/3)) -- the README combines a 3-point DCT with a
 *            64-point Hadamard matrix for d = 192;
 *
 * then y is quantised exactly as zyfa_fp8_quantize does (power-of-two
 * descale from max|y|, round to nearest even, saturating).  R is orthogonal,
 * so rotating q and k with the same signs leaves q k^T unchanged.  The
 * rotation is evaluated in FP32 (butterflies across the lanes of a warp).
 * Both kernels stream x in tiles of 64 rows through tensor-memory-access
 * copies; their waits are bounded like the attention kernel's and report
 * through zyfa_device_status().
 *
 * x          device, n_rows * d elements of x_dtype (ZYFA_BF16 or ZYFA_F32),
 *            rows contiguous, 16-byte aligned.
 * n_rows     number of rows (tokens x heads), >= 0; above 2^31 - 65
 *            (row coordinates of the copies are 32-bit) the call returns
 *            ZYFA_ERR_UNSUPPORTED.
 * d          128 or 192 (others: ZYFA_ERR_UNSUPPORTED).
 * signs      device, d FP32 values, each +1 or -1 (the same for q and k),
 *            4-byte aligned.
 * x8         device, n_rows * d codes, 16-byte aligned (rows are written
 *            as 16-byte chunks).
 * descale, workspace, stream: as for zyfa_fp8_quantize; deterministic (no
 *            atomics).
 * Returns ZYFA_OK or a negative zyfa_status (checks run before any launch).
 */
ZYFA_API int zyfa_fp8_quantize_rotated(const void* x, long long n_rows, int d, int x_dtype,
                                       const float* signs, void* x8, float* descale,
                                       void* workspace, struct CUstream_st* stream);

/* ABI version, (major << 16) | minor. */
ZYFA_API int zyfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZYFA_H */
