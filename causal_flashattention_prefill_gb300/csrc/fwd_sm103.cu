// Causal prefill attention forward for sm_103a (GB300).
//
// Computes O = softmax(scale * Q K^T + causal mask) V and the natural-log
// LSE of each row of scaled scores, the operation the ZYFA README defines
// ("Usage", "Supported configurations": causal forward pass, seqlen_q =
// seqlen_k, MHA/GQA/MQA, d_qk = d_v = 128 or d_qk = 192 with d_v = 128,
// BF16 or FP8 e4m3 inputs with one descale per tensor, BF16 output).
//
// One CTA per SM, persistent (or, with the dynamic schedule, one CTA per
// work item, of which about one per SM runs and takes the items of CTAs that
// have not started).  A work item is one query block of 256 rows (two
// 128-row tiles, "stage 0" and "stage 1") of one (batch, head).  Both
// tiles share every K/V tile that the CTA streams, so each K/V byte brought
// on chip serves 256 query rows (the wider-query-tile idea of the CDNA4 post,
// section 4.2, realised here as two tensor-memory accumulators).
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax of stage 0  (thread = query row = TMEM lane)
//   warps 4-7  softmax of stage 1
//   warp  8    TMA producer: Q tiles and a ring of K/V tiles (whole-tile
//              slots, or 16 KB pieces for BF16 d_qk = 192)
//   warp  9    MMA issuer: S = Q K^T (SS form) and O += P V (TS form, P read
//              from tensor memory, V as an MN-major operand); it learns that
//              a stage's P is ready on hardware barrier 1 + stage
//   warps 10-11 idle (they complete the third warpgroup so that registers
//              can move to the softmax warpgroups with setmaxnreg)
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   [0,128) S0   [128,256) S1   [256,384) O0   [384,512) O1
// P of a stage is written over the first columns of that stage's S.
//
// Online softmax (FlashAttention-2 tiling; ZYFA README "Kernel design"):
// exp2 with scale*log2(e) folded into one multiply-add, a reference maximum
// per row that moves only when the row maximum exceeds it by more than tau
// (lazy rescaling), and causal masking only on the diagonal tile.  Tiles
// above the diagonal are never loaded or computed.  Keys and queries past the
// end of the sequence read TMA's zero fill; the causal mask already hides
// such keys from every real query, which is the exact equivalent of padding
// the sequence with zeros (ZYFA README, "Usage").
#include <atomic>

#include <cuda_bf16.h>

#include "fwd.h"
#include "zyfa_ptx.cuh"

namespace zyfa {

__device__ int g_zyfa_status;

namespace {

constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Register split (setmaxnreg): the launch gives 384 x 168 = 64512 registers;
// the two softmax warpgroups take kSoftmaxRegs per thread and the third
// warpgroup (producer, MMA issuer, two idle warps) kOtherRegs, with
// 2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= 64512 (checked per config).
constexpr int kLaunchRegs = 168;
constexpr int kBM = 128;  // query rows per stage
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kDV = 128;
constexpr int kMaxDynSmem = 232448;

// 2^n as a float, for compile-time constants.
constexpr float exp2i(int n) {
  float r = 1.0f;
  for (int i = 0; i < n; ++i) r *= 2.0f;
  return r;
}

template <int DT, int DQK, int RP = 0, int BS = 0>
struct Cfg {
  static constexpr bool kF8 = DT == 1;
  // BS (FP8): per-block scaling of P (ZYFA README, "Kernel design",
  // per-block scaling).  Each row's P is scaled per 32-key slice by the
  // power of two that brings the slice's largest value to the binade of
  // p = 1, so that small probabilities stay normal e4m3 values, and the P V
  // product is the block-scaled MMA (kind::mxf8f6f4), which multiplies each
  // slice by the inverse power of two (a UE8M0 scale factor per row and
  // slice) as it accumulates.
  static constexpr bool kBlockScale = BS != 0;
  static_assert(!kBlockScale || kF8, "block scaling is an FP8 form");
  // RP: the denominator of O is, on every tile, the sum of the rounded P
  // values that multiply V (BF16 values; FP8 e4m3 codes, plus the lo term
  // where the tile has one), so each output row is a weighted average whose
  // weights sum to one (ZYFA README, "Accuracy").  Without RP that sum is
  // taken only where one probability carries a large share of the row's
  // mass, and the unrounded sum stands in elsewhere.
  static constexpr bool kRoundedP = RP != 0;
  static constexpr int kElem = kF8 ? 1 : 2;
  // Q and K: rows of DQK elements, stored as column chunks of one swizzle
  // span each (128 bytes, or 64 bytes when the row is not a multiple of 128).
  static constexpr int kRowBytesQK = DQK * kElem;
  static constexpr int kSwzQK = (kRowBytesQK % 128 == 0) ? 128 : 64;
  static constexpr uint32_t kSwzModeQK = kSwzQK == 128 ? 2u : 4u;
  static constexpr int kChunkElemsQK = kSwzQK / kElem;
  static constexpr int kChunksQK = kRowBytesQK / kSwzQK;
  static constexpr int kChunkBytesQK = kBM * kSwzQK;
  static constexpr int kTileBytesQK = kChunksQK * kChunkBytesQK;
  // V: rows of 128 elements in 128-byte chunks.
  static constexpr int kChunkElemsV = 128 / kElem;
  static constexpr int kChunksV = kDV * kElem / 128;
  static constexpr int kChunkBytesV = kBN * 128;
  static constexpr int kTileBytesV = kChunksV * kChunkBytesV;
  static constexpr int kSlotBytes = kTileBytesQK > kTileBytesV ? kTileBytesQK : kTileBytesV;
  static constexpr int kUmmaK = 32 / kElem;   // reduction depth of one MMA
  static constexpr int kReserve = 2048;       // alignment slack + barriers
  static constexpr int kSlotsFit = (kMaxDynSmem - kReserve - 2 * kTileBytesQK) / kSlotBytes;
  static constexpr int kNumSlots = kSlotsFit > 8 ? 8 : kSlotsFit;
  // The K/V ring is a FIFO of pieces; a K tile takes kPiecesK consecutive
  // pieces and a V tile kPiecesV.  Where whole-tile slots would leave no
  // room to load ahead (fewer than three fit: BF16 d_qk = 192, whose Q tiles
  // take 96 KB), a piece is one 16 KB chunk of a tile (128 rows x 128 bytes),
  // so the next tiles start loading while the current ones are in use;
  // elsewhere a piece is a whole-tile slot.
  static constexpr bool kChunkPieces = kSlotsFit < 3;
  static constexpr int kPieceBytes = kChunkPieces ? 128 * 128 : kSlotBytes;
  static constexpr int kCppK = kChunkPieces ? 1 : kChunksQK;  // K chunks per piece
  static constexpr int kCppV = kChunkPieces ? 1 : kChunksV;   // V chunks per piece
  static constexpr int kPiecesK = kChunksQK / kCppK;
  static constexpr int kPiecesV = kChunksV / kCppV;
  static constexpr int kPiecesFit = (kMaxDynSmem - kReserve - 2 * kTileBytesQK) / kPieceBytes;
  static constexpr int kNumPieces =
      kChunkPieces ? (kPiecesFit > 8 ? 8 : kPiecesFit) : kNumSlots;
  static constexpr int kSmemBytes = kReserve + 2 * kTileBytesQK + kNumPieces * kPieceBytes;
  // Lazy-rescale threshold in base-2 units of the score (the ZYFA README's
  // "Kernel design" uses 0.125-8).  Large thresholds keep the reference
  // from moving after the first tiles, so exp2 can run against it before
  // the tile maximum is known: BF16 16 (p <= 2^16, far inside BF16 and the
  // FP32 sums and accumulators), FP8 6 (p * 2^2 <= 256, inside e4m3's 448).
  // With block scaling, P never exceeds 8 (each slice is normalised), so
  // FP8 takes the BF16 threshold.
  static constexpr int kTauBits = (kF8 && !kBlockScale) ? 6 : 16;
  static constexpr float kTau = static_cast<float>(kTauBits);
  // FP8 P is stored as e4m3 of p * 2^2 (p <= 2^tau keeps it below 448); the
  // factor enters as +2 in the exponent.  (A pre-scale of 2^4 with tau 4
  // keeps probabilities two binades further down from underflow; 2^2 with
  // tau 6 rescales less often and measured 1 % faster, and the smallest
  // probability kept, 2^-12 of the reference, is far below what the
  // stated tolerances can see.)
  static constexpr int kPLog2Bits = kF8 ? 2 : 0;
  static constexpr float kPLog2Scale = static_cast<float>(kPLog2Bits);
  // Largest p that needs no rescale: 2^(tau + pre-scale).
  static constexpr float kPCap = exp2i(kTauBits + kPLog2Bits);
  // Accuracy test: a p above 1/kAccRatio of the row's mass so far takes the
  // exact path (BF16 rounded-sum denominator, FP8 two-term P).  FP8 with the
  // rounded-P denominator keeps 1/32: its LSE mode sums the rounded values,
  // whose error the two-term tiles bound.
  static constexpr float kAccRatio = kF8 ? (kRoundedP ? 32.0f : 16.0f) : 8.0f;
  static constexpr uint32_t kFmt = kF8 ? 0u : 1u;   // E4M3 / BF16
  static constexpr uint32_t kIdescQK = ptx::instr_desc(kFmt, kFmt, 0, kBM, kBN);
  static constexpr uint32_t kIdescPV = ptx::instr_desc(kFmt, kFmt, 1, kBM, kDV);
  // Block-scaled P V, K slice ks (one MMA): byte ks of the scale-factor words.
  __host__ __device__ static constexpr uint32_t idesc_pv_bs(int ks) {
    return ptx::instr_desc_bs(0u, 0u, 1u, kBM, kDV, static_cast<uint32_t>(ks),
                              static_cast<uint32_t>(ks));
  }
  // Register split: the MMA issuer of the d_qk = 192 BF16 form unrolls 12
  // K steps and needs more registers than the others.
  static constexpr int kSoftmaxRegs = (!kF8 && DQK == 192) ? 184 : 200;
  // The MMA issuer's loop over the two stages is kept rolled (half the
  // issuer code) except for BF16 d_qk = 128, where the unrolled loop
  // measured faster; rolled, the FP8 and d_qk = 192 forms measured 5-12 %
  // faster on activation-like rows and short sequences.
  static constexpr bool kRollStages = kF8 || DQK == 192;
  // BF16 d_qk = 128: the speculative pass keeps one sum per 32-key chunk,
  // whose largest bounds the tile's p in the quiet test (about 4x tighter
  // than the tile sum on flat rows; measured slower on the d_qk = 192 form).
  static constexpr bool kChunkBound = !kF8 && DQK == 128;
  static_assert(kRollStages || (!kF8 && kSlotsFit >= 3),
                "the unrolled stage loop carries neither the FP8 residual P V nor the piece ring");
  static constexpr int kOtherRegs = (!kF8 && DQK == 192) ? 136 : 104;
  static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static_assert(kNumSlots >= 2, "K/V ring needs at least two slots");
  static_assert(!kChunkPieces || (kChunkBytesQK == kPieceBytes && kChunkBytesV == kPieceBytes),
                "chunk pieces hold one chunk each");
  static_assert(kNumPieces >= kPiecesK + 2 * kPiecesV,
                "ring holds a V tile, the next K tile and a V tile with a skipped piece");
  static_assert(kNumPieces <= 8, "ring bookkeeping packs 4 bits per piece");
  static_assert(kSmemBytes <= kMaxDynSmem, "shared memory budget");
  static_assert(kPieceBytes % 1024 == 0 && kTileBytesQK % 1024 == 0, "1 KB alignment");
};

struct Item {
  int b, h, u;
  int n0, n1;     // K/V tiles processed by stage 0 and stage 1 (0 = stage idle)
  int nload;      // K/V tiles loaded = max(n0, n1)
};

// Items (numbered longest first, see decode_item) reach a CTA in one of two
// ways.  Static (default): a grid of min(items, SMs) CTAs; CTA c of G takes,
// in round r, item r*G + c for even r and r*G + G-1-c for odd r (a
// serpentine deal that evens out the decreasing costs).  Dynamic
// (ZYFA_OPT_DYNAMIC_SCHEDULE): one CTA per item; a running CTA takes the
// items of CTAs that have not started by cancelling them (cluster launch
// control), so the longest remaining item goes to whichever SM frees up
// first -- better where item costs vary with the data, slightly worse on
// regular rows; the producer warp makes the requests and passes the item
// sequence to the MMA issuer and the softmax warps through a ring of
// kItemRing slots (in the static schedule every warp computes it).
__device__ __forceinline__ int item_index(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? (grid - 1 - cta) : cta);
}

constexpr int kItemRing = 4;
constexpr int kItemConsumers = 9;   // the MMA issuer warp and eight softmax warps

// Item w, the w-th longest: query block u descending, then batch, then head
// (so the query heads of one KV group run side by side and share K/V in
// L2).  Stage 0 (tile 2u) needs K/V tiles 0..2u; stage 1 (tile 2u+1) needs
// 0..2u+1 and is idle when all its rows lie past the sequence end.
__device__ __forceinline__ Item decode_item(int w, const FwdParams& p) {
  Item it;
  const int per_block = p.B * p.H;
  const int r = w / per_block;
  const int rem = w - r * per_block;
  it.u = p.n_qblocks - 1 - r;
  it.b = rem / p.H;
  it.h = rem - it.b * p.H;
  it.n0 = 2 * it.u + 1;
  it.n1 = (kBM * (2 * it.u + 1) < p.S) ? 2 * it.u + 2 : 0;
  it.nload = it.n1 > it.n0 ? it.n1 : it.n0;
  return it;
}

struct Smem {
  uint8_t* q[2];
  uint8_t* slots;
  uint64_t* bars;
  uint32_t* tmem_base;
  int* abort;
  volatile uint32_t* pflag;   // [stage]: index of the last tile with a two-term FP8 P
  volatile int* items;        // [kItemRing]: item sequence (-1: no more items)
  uint32_t clc_resp;          // shared-memory address of the 16-byte cancel response
};

// Barrier indices inside the barrier array.
template <int NS>
struct Bars {
  static constexpr int kQFull = 0;            // [2]
  static constexpr int kQEmpty = 2;           // [2]
  static constexpr int kSFull = 4;            // [2]
  static constexpr int kOFull = 6;            // [2]
  static constexpr int kDrain = 8;
  static constexpr int kPvDone = 9;           // [2]
  static constexpr int kItemFull = 11;        // [kItemRing]
  static constexpr int kItemEmpty = 15;       // [kItemRing]
  static constexpr int kClc = 19;             // cancel response landed
  static constexpr int kSlotFull = 20;        // [NS]
  static constexpr int kSlotEmpty = 20 + NS;  // [NS]
  static constexpr int kCount = 20 + 2 * NS;
};

// Placement of K/V tiles in the ring.  The producer and the MMA issuer walk
// the same tile sequence (K_0, then V_j and K_j+1 for each step j, item
// after item) and place each tile with this, so they agree on every piece.
// Pieces are taken in cyclic order and released in the same order.
template <class C>
struct Ring {
  uint32_t pc = 0;  // next free piece
  // Places a K tile (v = false) or a V tile (v = true).  Returns its first
  // occupied piece, whose full and empty barriers the tile uses; `base` is
  // the piece of its chunk 0 and `last` its last occupied piece.  The chunks
  // of a V tile are one MMA operand with a fixed stride, so a V tile that
  // would wrap around the ring skips to piece 0 and keeps the skipped
  // pieces; K chunks are separate operands and may wrap.
  __device__ __forceinline__ uint32_t place(bool v, uint32_t& base, uint32_t& last) {
    constexpr uint32_t np = C::kNumPieces;
    const uint32_t n = v ? C::kPiecesV : C::kPiecesK;
    const uint32_t first = pc;
    base = (v && pc + n > np) ? 0u : pc;
    pc = base + n;
    if (pc >= np) pc -= np;            // base + n < 2 np: no division
    last = pc == 0 ? np - 1 : pc - 1;
    return first;
  }
  // Shared-memory byte offset (from the ring start) of chunk c of a tile
  // whose chunk 0 is in piece `base` (c a compile-time constant at every
  // call site, so the slot form is one multiply-add).
  static __device__ __forceinline__ uint32_t k_chunk(uint32_t base, int c) {
    if constexpr (!C::kChunkPieces) {
      return base * C::kPieceBytes + c * C::kChunkBytesQK;
    } else {
      uint32_t q = base + c;
      if (q >= C::kNumPieces) q -= C::kNumPieces;
      return q * C::kPieceBytes;
    }
  }
  static __device__ __forceinline__ uint32_t v_chunk(uint32_t base, int c) {
    return (base + c / C::kCppV) * C::kPieceBytes + (c % C::kCppV) * C::kChunkBytesV;
  }
};

__device__ __forceinline__ void tma_tile(const CUtensorMap* m, uint32_t dst, uint32_t bar,
                                         int layout, int c0, int head, int row, int b,
                                         uint64_t pol) {
  if (layout == 0)
    ptx::tma_load_4d(dst, m, bar, c0, head, row, b, pol);
  else
    ptx::tma_load_4d(dst, m, bar, c0, row, head, b, pol);
}

// Waits for a phase with the whole warp: the warp leaves the wait
// converged and in agreement, as the .sync.aligned tcgen05 instructions that
// follow require.
__device__ __forceinline__ bool warp_wait(uint32_t b, uint32_t parity, volatile int* abort,
                                          int* status, int lane) {
  // Common case: every lane sees the completed phase (one vote, no
  // divergence).  Otherwise one lane waits with the timeout and the verdict
  // is broadcast.
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(b, parity))) return true;
  int ok = 0;
  if (lane == 0) ok = ptx::mbar_wait(b, parity, abort, status, 1) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  // Each lane observes the completed phase itself (an acquire of its own);
  // the phase cannot move on before this warp's next arrival.
  if (ok) (void)ptx::mbar_test(b, parity);
  return ok != 0;
}

// Maximum of 64 / 128 scores: independent chains of three-input max.
__device__ __forceinline__ float row_max64(const float* f) {
  float m4[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float acc = ptx::max3(f[16 * a], f[16 * a + 1], f[16 * a + 2]);
#pragma unroll
    for (int k = 3; k < 15; k += 2) acc = ptx::max3(acc, f[16 * a + k], f[16 * a + k + 1]);
    m4[a] = fmaxf(acc, f[16 * a + 15]);
  }
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

__device__ __forceinline__ float row_max128(const float* f) {
  return fmaxf(row_max64(f), row_max64(f + 64));
}

// Maximum of 32 scores (two chains of three-input max).
__device__ __forceinline__ float row_max32(const float* f) {
  float a = ptx::max3(f[0], f[1], f[2]);
  float b = ptx::max3(f[3], f[4], f[5]);
#pragma unroll
  for (int k = 6; k < 30; k += 4) {
    a = ptx::max3(a, f[k], f[k + 1]);
    b = ptx::max3(b, f[k + 2], f[k + 3]);
  }
  return ptx::max3(a, b, fmaxf(f[30], f[31]));
}

// Tensor-memory columns of a stage's S region that hold, once the softmax
// has read S, the scale factors of the block-scaled P V: those of P (one
// 32-bit word per row, byte k for key slice k; the rows of lane quarter q
// in column kSfaCol + q) and those of V (all 2^0).
constexpr uint32_t kSfaCol = 64;
constexpr uint32_t kSfbCol = 96;

// Exponent e of the power of two 2^e that brings the largest P of a 32-key
// slice, 2^y with y = (slice maximum) * c - m_ref, into the binade of p = 1:
// e = -floor(y), kept within [-32, 100] (an entirely masked slice has
// y = -inf; its P is zero under any scale).
__device__ __forceinline__ float slice_exponent(float xm, float c_log2, float m_ref) {
  const float y = fmaf(xm, c_log2, -m_ref);
  return fminf(fmaxf(-floorf(y), -32.0f), 100.0f);
}

// 2^-e for an integral e in [-32, 100], exactly.
__device__ __forceinline__ float pow2_neg(float e) {
  return __int_as_float((127 - static_cast<int>(e)) << 23);
}

// O of the row times alpha, in tensor memory.  (The scores stay live
// across a rescale, so O goes through 32 registers at a time.)
__device__ __forceinline__ void rescale_o(uint32_t t_o, float alpha) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    ptx::tmem_ld32_wait(t_o + c * 32, o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
    ptx::tmem_st32(t_o + c * 32, o);
  }
}

// P for 64 scores (half h of the row): p = 2^(s*c + neg_m) by paired FMAs
// and exp2, packed to BF16 (or e4m3; with two_term also the e4m3 rounding
// residual at column offset 32), stored to tensor memory over S.  `sacc`
// accumulates the unrounded sum; with kExact (BF16) `rr` accumulates the sum
// of the rounded values that multiply V.
// kTest (FP8): every packed word of P also enters the threshold test
// tacc |= word + tk (see threshold_addend).
template <class C, bool kExact, bool kTest = false>
__device__ __forceinline__ void produce_half(const float* f, float c_log2, float neg_m,
                                             uint32_t t_s, int h, bool two_term,
                                             float2 (&sacc)[2], float& rr, uint32_t tk = 0,
                                             uint32_t* tacc = nullptr, int cc0 = 0,
                                             int ncc = 2, float* csum = nullptr) {
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
  for (int cc = cc0; cc < cc0 + ncc; ++cc) {
    const int ch = 2 * h + cc;  // 32-column chunk of the row
    float e[32];
    float2 cacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 (&acc)[2] = csum ? cacc : sacc;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 x = __ffma2_rn(make_float2(f[32 * ch + 2 * i], f[32 * ch + 2 * i + 1]), c2, nm2);
      e[2 * i] = ptx::ex2(x.x);
      e[2 * i + 1] = ptx::ex2(x.y);
      acc[i & 1] = __fadd2_rn(acc[i & 1], make_float2(e[2 * i], e[2 * i + 1]));
    }
    if (csum) {
      const float2 t = __fadd2_rn(cacc[0], cacc[1]);
      csum[ch] = t.x + t.y;
    }
    if constexpr (C::kF8) {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pk[i] = ptx::pack_e4m3x4(e[4 * i], e[4 * i + 1], e[4 * i + 2], e[4 * i + 3]);
      ptx::tmem_st8(t_s + ch * 8, pk);
      if constexpr (kTest) {
#pragma unroll
        for (int i = 0; i < 8; ++i) *tacc |= pk[i] + tk;
      }
      if constexpr (C::kRoundedP) {
        float a2[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 8; ++i) a2[i & 1] = ptx::add_e4m3x4_f32(a2[i & 1], pk[i]);
        rr += a2[0] + a2[1];
      }
      if (two_term) {
        uint32_t lo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float d[4];
          ptx::unpack_e4m3x4(pk[i], d);
          lo[i] = ptx::pack_e4m3x4(e[4 * i] - d[0], e[4 * i + 1] - d[1], e[4 * i + 2] - d[2],
                                   e[4 * i + 3] - d[3]);
        }
        ptx::tmem_st8(t_s + 32 + ch * 8, lo);
        if constexpr (C::kRoundedP) {
          float a2[2] = {0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 8; ++i) a2[i & 1] = ptx::add_e4m3x4_f32(a2[i & 1], lo[i]);
          rr += a2[0] + a2[1];
        }
      }
    } else {
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16x2(e[2 * i], e[2 * i + 1]);
      ptx::tmem_st16(t_s + ch * 16, pk);
      if constexpr (kExact || C::kRoundedP) {
        float a2[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) a2[i & 1] = ptx::add_bf16x2_f32(a2[i & 1], pk[i]);
        rr += a2[0] + a2[1];
      }
    }
  }
}

// FP8 threshold test on packed P.  The e4m3 code of a non-negative value is
// monotonic in the value and at most 0x7E, so adding 0x80 - c to every byte
// of a word sets that byte's top bit exactly when its code is >= c, without
// carries between bytes.  Returns the per-byte addend for code c.
__device__ __forceinline__ uint32_t threshold_addend(uint32_t c) {
  return (0x80u - c) * 0x01010101u;
}

// FP8: the lo term of the row's P (the e4m3 rounding residual of hi, stored
// at column offset 32 of S), and with do_hi also the hi term and its
// unrounded sum rs, from one exp2 pass (hi and rs are the values, in the
// same order, that produce_tile gives).  Without do_hi the hi codes in
// tensor memory are those this pass would store.
//   With kRoundedP the sum of the rounded values that multiply V is also
// formed: rr becomes the sum of hi and lo with do_hi, and gains the sum of
// lo without (the hi codes then being those already summed).
template <class C>
__device__ __forceinline__ void redo_fp8(const float* f, float c_log2, float neg_m,
                                         uint32_t t_s, bool do_hi, float& rs, float& rr) {
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(neg_m, neg_m);
  float2 sacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float ra[2] = {0.f, 0.f};
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 xa =
          __ffma2_rn(make_float2(f[32 * ch + 4 * i], f[32 * ch + 4 * i + 1]), c2, nm2);
      const float2 xb =
          __ffma2_rn(make_float2(f[32 * ch + 4 * i + 2], f[32 * ch + 4 * i + 3]), c2, nm2);
      const float e0 = ptx::ex2(xa.x), e1 = ptx::ex2(xa.y), e2 = ptx::ex2(xb.x),
                  e3 = ptx::ex2(xb.y);
      if (do_hi) {
        sacc[0] = __fadd2_rn(sacc[0], make_float2(e0, e1));
        sacc[1] = __fadd2_rn(sacc[1], make_float2(e2, e3));
      }
      hi[i] = ptx::pack_e4m3x4(e0, e1, e2, e3);
      float d[4];
      ptx::unpack_e4m3x4(hi[i], d);
      lo[i] = ptx::pack_e4m3x4(e0 - d[0], e1 - d[1], e2 - d[2], e3 - d[3]);
    }
    if (do_hi) ptx::tmem_st8(t_s + ch * 8, hi);
    ptx::tmem_st8(t_s + 32 + ch * 8, lo);
    if constexpr (C::kRoundedP) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (do_hi) ra[i & 1] = ptx::add_e4m3x4_f32(ra[i & 1], hi[i]);
        ra[i & 1] = ptx::add_e4m3x4_f32(ra[i & 1], lo[i]);
      }
    }
  }
  if (do_hi) {
    const float2 t2 = __fadd2_rn(sacc[0], sacc[1]);
    rs = t2.x + t2.y;
  }
  if constexpr (C::kRoundedP) rr = (do_hi ? 0.f : rr) + (ra[0] + ra[1]);
}

// BF16: the sum rr of the rounded P of the row (the values that multiply
// V), and with do_hi also P itself (stored over S) and its unrounded sum rs,
// from one exp2 pass (P and rs are the values, in the same order, that
// produce_tile gives).  Without do_hi the P in tensor memory is the one this
// pass would store.
__device__ __forceinline__ void redo_bf16(const float* f, float c_log2, float neg_m,
                                          uint32_t t_s, bool do_hi, float& rs, float& rr) {
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(neg_m, neg_m);
  float2 sacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int q = 16 * ch + i;  // pair index in the row
      const float2 x = __ffma2_rn(make_float2(f[2 * q], f[2 * q + 1]), c2, nm2);
      const float e0 = ptx::ex2(x.x), e1 = ptx::ex2(x.y);
      if (do_hi) sacc[i & 1] = __fadd2_rn(sacc[i & 1], make_float2(e0, e1));
      pk[i] = ptx::pack_bf16x2(e0, e1);
      a[q & 3] = ptx::add_bf16x2_f32(a[q & 3], pk[i]);
    }
    if (do_hi) ptx::tmem_st16(t_s + ch * 16, pk);
  }
  rr = (a[0] + a[1]) + (a[2] + a[3]);
  if (do_hi) {
    const float2 t2 = __fadd2_rn(sacc[0], sacc[1]);
    rs = t2.x + t2.y;
  }
}

// FP8 with per-slice scales: for key slice k of the row, P' = 2^(s*c + neg_m
// + e_k) (the slice's largest value in [4, 8), the binade of the code of
// p = 1 times the pre-scale, when the slice is not
// clamped), hi codes stored at column 8k and with kLo the e4m3 rounding
// residual at 32 + 8k.  With kHi, rs = the unrounded sum of P = P' 2^-e_k
// over the row.  With kRoundedP, rr gains the sum of the rounded values
// that multiply V (hi with kHi, lo with kLo), each slice times 2^-e_k.
// Without kHi the pass recomputes hi only to form lo (the hi codes in
// tensor memory are those it would store).
template <class C, bool kHi, bool kLo>
__device__ __forceinline__ void produce_bs(const float* f, float c_log2, float neg_m,
                                           const float (&ex)[4], uint32_t t_s, float& rs,
                                           float& rr) {
  const float2 c2 = make_float2(c_log2, c_log2);
  float rsum = 0.f;
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    const float bias = neg_m + ex[ch];
    const float2 b2 = make_float2(bias, bias);
    const float down = pow2_neg(ex[ch]);
    float2 sacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 xa =
          __ffma2_rn(make_float2(f[32 * ch + 4 * i], f[32 * ch + 4 * i + 1]), c2, b2);
      const float2 xb =
          __ffma2_rn(make_float2(f[32 * ch + 4 * i + 2], f[32 * ch + 4 * i + 3]), c2, b2);
      const float e0 = ptx::ex2(xa.x), e1 = ptx::ex2(xa.y), e2 = ptx::ex2(xb.x),
                  e3 = ptx::ex2(xb.y);
      if constexpr (kHi) {
        sacc[0] = __fadd2_rn(sacc[0], make_float2(e0, e1));
        sacc[1] = __fadd2_rn(sacc[1], make_float2(e2, e3));
      }
      hi[i] = ptx::pack_e4m3x4(e0, e1, e2, e3);
      if constexpr (kLo) {
        float d[4];
        ptx::unpack_e4m3x4(hi[i], d);
        lo[i] = ptx::pack_e4m3x4(e0 - d[0], e1 - d[1], e2 - d[2], e3 - d[3]);
      }
    }
    if constexpr (kHi) ptx::tmem_st8(t_s + ch * 8, hi);
    if constexpr (kLo) ptx::tmem_st8(t_s + 32 + ch * 8, lo);
    if constexpr (kHi) {
      const float2 t2 = __fadd2_rn(sacc[0], sacc[1]);
      rsum += (t2.x + t2.y) * down;
    }
    if constexpr (C::kRoundedP) {
      float a2[2] = {0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if constexpr (kHi) a2[i & 1] = ptx::add_e4m3x4_f32(a2[i & 1], hi[i]);
        if constexpr (kLo) a2[i & 1] = ptx::add_e4m3x4_f32(a2[i & 1], lo[i]);
      }
      rr += (a2[0] + a2[1]) * down;
    }
  }
  if constexpr (kHi) rs = rsum;
}

// P for the whole 128-score row against reference neg_m; rs = unrounded
// sum, rr = sum of the rounded values (with kRR, BF16).  The variant is a
// template argument so that each call site carries only the code it runs.
template <class C, bool kRR>
__device__ __forceinline__ void produce_tile(const float* f, float c_log2, float neg_m,
                                             uint32_t t_s, bool two_term, float& rs, float& rr) {
  float2 sacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  rr = 0.f;
  produce_half<C, kRR>(f, c_log2, neg_m, t_s, 0, two_term, sacc, rr);
  produce_half<C, kRR>(f, c_log2, neg_m, t_s, 1, two_term, sacc, rr);
  const float2 t2 = __fadd2_rn(sacc[0], sacc[1]);
  rs = t2.x + t2.y;
}

}  // namespace

template <int DT, int DQK, int RP, int BS, int DS>
__global__ void __launch_bounds__(kThreads, 1)
    zyfa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<DT, DQK, RP, BS>;
  constexpr bool kDynamic = DS != 0;   // dynamic schedule (see item_index)
  constexpr int NS = C::kNumPieces;
  using B = Bars<NS>;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Smem sm;
  sm.q[0] = base;
  sm.q[1] = base + C::kTileBytesQK;
  sm.slots = base + 2 * C::kTileBytesQK;
  sm.bars = reinterpret_cast<uint64_t*>(sm.slots + NS * C::kPieceBytes);
  sm.tmem_base = reinterpret_cast<uint32_t*>(sm.bars + B::kCount);
  sm.abort = reinterpret_cast<int*>(sm.tmem_base + 1);
  sm.pflag = reinterpret_cast<volatile uint32_t*>(sm.abort + 1);
  sm.items = reinterpret_cast<volatile int*>(sm.pflag + 2);
  sm.clc_resp = (ptx::smem_u32(const_cast<int*>(sm.items) + kItemRing) + 15u) & ~15u;
  volatile int* abort = sm.abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bars_smem = ptx::smem_u32(sm.bars);
  const uint32_t q_smem = ptx::smem_u32(sm.q[0]);
  const uint32_t slots_smem = ptx::smem_u32(sm.slots);
  auto bar = [&](int i) { return bars_smem + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B::kQFull + 0), 1);
    ptx::mbar_init(bar(B::kQFull + 1), 1);
    ptx::mbar_init(bar(B::kQEmpty + 0), 1);
    ptx::mbar_init(bar(B::kQEmpty + 1), 1);
    ptx::mbar_init(bar(B::kSFull + 0), 1);
    ptx::mbar_init(bar(B::kSFull + 1), 1);
    ptx::mbar_init(bar(B::kOFull + 0), 1);
    ptx::mbar_init(bar(B::kOFull + 1), 1);
    ptx::mbar_init(bar(B::kDrain), 1);
    ptx::mbar_init(bar(B::kPvDone + 0), 1);
    ptx::mbar_init(bar(B::kPvDone + 1), 1);
    for (int i = 0; i < kItemRing; ++i) {
      ptx::mbar_init(bar(B::kItemFull + i), 1);
      ptx::mbar_init(bar(B::kItemEmpty + i), kItemConsumers);
    }
    ptx::mbar_init(bar(B::kClc), 1);
    for (int i = 0; i < NS; ++i) {
      ptx::mbar_init(bar(B::kSlotFull + i), 1);
      ptx::mbar_init(bar(B::kSlotEmpty + i), 1);
    }
    *sm.abort = 0;
    sm.pflag[0] = 0;
    sm.pflag[1] = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  __syncwarp();
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(sm.tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *sm.tmem_base;

  int* status = &g_zyfa_status;
  // Item r of this CTA's sequence for a consuming warp (the MMA issuer or a
  // softmax warp), -1 after the last: computed in the static schedule; in
  // the dynamic one, read from the producer's slot, which is then released.
  auto take_item = [&](int r, int& w) -> bool {
    if constexpr (!kDynamic) {
      w = item_index(r, blockIdx.x, gridDim.x);
      if (w >= p.total_items) w = -1;
      return true;
    } else {
      const int slot = r & (kItemRing - 1);
      if (!warp_wait(bar(B::kItemFull + slot), static_cast<uint32_t>(r / kItemRing) & 1u, abort,
                     status, lane))
        return false;
      w = sm.items[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(B::kItemEmpty + slot));
      return true;
    }
  };

  // Each setmaxnreg sits inside its role's branch so that the register
  // allocator sees the softmax code only on the 224-register path.
  if (warp >= 8) {
    ptx::setmaxnreg_dec<C::kOtherRegs>();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      uint32_t q_par = 0;   // bit s: parity of the uses of Q buffer s so far
      uint32_t q_used = 0;  // bit s: Q buffer s was loaded at least once
      uint32_t t = 0;       // slot ring: K/V tiles issued so far (ring position)
      Ring<C> ring;         // chunk-piece ring: placement
      // Slot ring: the MMA issuer consumes the tiles in units: K_0 alone,
      // then (V_j, K_j+1) in step j.  Each unit completes on the full barrier
      // of its first tile (armed with the bytes of the whole unit), so the
      // issuer waits once per step.  fpar bit x: phase parity of full
      // barrier x after its last arming; armed bit x: armed at least once.
      uint32_t fpar = 0, armed = 0;
      uint32_t unit_bar = 0;
      // Piece ownership: the tile that last took piece q releases it on the
      // empty barrier own_b[q] (4 bits per piece) with phase parity
      // own_par bit q; own_valid bit q: piece q was ever taken.  rel_par bit
      // x: parity of the next release phase of empty barrier x.  Pieces are
      // taken and released in the same cyclic order, so a tile needs only
      // the release of the newest earlier owner among its pieces: the owner
      // of its last piece.
      uint32_t own_b = 0, own_par = 0, own_valid = 0, rel_par = 0;
      const int group = p.H / p.Hkv;
      bool ok = true;
      int w = blockIdx.x;       // this CTA's own item first
      bool more = true;
      uint32_t clc_par = 0;
      bool clc_pending = false;
      for (int r = 0; ok; ++r) {
        if constexpr (kDynamic) {
          // Item r (or the end) to the MMA issuer and the softmax warps.
          const int islot = r & (kItemRing - 1);
          if (r >= kItemRing) {
            ok = ptx::mbar_wait(bar(B::kItemEmpty + islot),
                                (static_cast<uint32_t>(r / kItemRing) & 1u) ^ 1u, abort, status,
                                1);
            if (!ok) break;
          }
          sm.items[islot] = more ? w : -1;
          ptx::mbar_arrive(bar(B::kItemFull + islot));
        }
        if (!more) break;
        const Item it = decode_item(w, p);
        const int nst = it.n1 > 0 ? 2 : 1;
        for (int s = 0; s < nst && ok; ++s) {
          ok = ptx::mbar_wait(bar(B::kQEmpty + s), ((q_par >> s) & 1u) ^ 1u, abort, status, 1);
          if (!ok) break;
          const uint32_t qb = bar(B::kQFull + s);
          ptx::mbar_arrive_expect_tx(qb, C::kTileBytesQK);
          const int row0 = (2 * it.u + s) * kBM;
          const uint32_t qdst = q_smem + s * C::kTileBytesQK;
#pragma unroll
          for (int c = 0; c < C::kChunksQK; ++c)
            tma_tile(&tm_q, qdst + c * C::kChunkBytesQK, qb, p.layout, c * C::kChunkElemsQK,
                     it.h, row0, it.b, pol_q);
          q_par ^= 1u << s;
          q_used |= 1u << s;
        }
        const int hk = it.h / group;
        if constexpr (!C::kChunkPieces) {
          for (int j = 0; j < it.nload && ok; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
              const uint32_t slot = t % NS;
              ok = ptx::mbar_wait(bar(B::kSlotEmpty + slot), ((t / NS) & 1u) ^ 1u, abort, status,
                                  1);
              if (!ok) break;
              const uint32_t dst = slots_smem + slot * C::kSlotBytes;
              if (kv == 0) {
                uint32_t fb = unit_bar;  // K_j, j > 0: second tile of the unit (V_j-1, K_j)
                if (j == 0) {
                  fb = bar(B::kSlotFull + slot);
                  ptx::mbar_arrive_expect_tx(fb, C::kTileBytesQK);
                  fpar ^= 1u << slot;
                  armed |= 1u << slot;
                }
  #pragma unroll
                for (int c = 0; c < C::kChunksQK; ++c)
                  tma_tile(&tm_k, dst + c * C::kChunkBytesQK, fb, p.layout,
                           c * C::kChunkElemsQK, hk, j * kBN, it.b, pol_kv);
              } else {
                const uint32_t fb = bar(B::kSlotFull + slot);
                ptx::mbar_arrive_expect_tx(
                    fb, C::kTileBytesV + (j + 1 < it.nload ? C::kTileBytesQK : 0));
                fpar ^= 1u << slot;
                armed |= 1u << slot;
                unit_bar = fb;
  #pragma unroll
                for (int c = 0; c < C::kChunksV; ++c)
                  tma_tile(&tm_v, dst + c * C::kChunkBytesV, fb, p.layout, c * C::kChunkElemsV,
                           hk, j * kBN, it.b, pol_kv);
              }
              ++t;
            }
          }
        } else {
          for (int j = 0; j < it.nload && ok; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
              uint32_t base, last;
              const uint32_t first = ring.place(kv == 1, base, last);
              if ((own_valid >> last) & 1u) {
                ok = ptx::mbar_wait(bar(B::kSlotEmpty + ((own_b >> (4 * last)) & 0xFu)),
                                    (own_par >> last) & 1u, abort, status, 1);
                if (!ok) break;
              }
              const uint32_t rp = (rel_par >> first) & 1u;
              rel_par ^= 1u << first;
              for (uint32_t q = first;; q = (q + 1 == NS) ? 0u : q + 1) {
                own_b = (own_b & ~(0xFu << (4 * q))) | (first << (4 * q));
                own_par = (own_par & ~(1u << q)) | (rp << q);
                own_valid |= 1u << q;
                if (q == last) break;
              }
              // Every tile completes on the full barrier of its first piece,
              // so the issuer starts P V_j while K_j+1 is still loading.
              const uint32_t fb = bar(B::kSlotFull + first);
              ptx::mbar_arrive_expect_tx(fb, kv == 0 ? C::kTileBytesQK : C::kTileBytesV);
              fpar ^= 1u << first;
              armed |= 1u << first;
              if (kv == 0) {
  #pragma unroll
                for (int c = 0; c < C::kChunksQK; ++c)
                  tma_tile(&tm_k, slots_smem + Ring<C>::k_chunk(base, c), fb, p.layout,
                           c * C::kChunkElemsQK, hk, j * kBN, it.b, pol_kv);
              } else {
  #pragma unroll
                for (int c = 0; c < C::kChunksV; ++c)
                  tma_tile(&tm_v, slots_smem + Ring<C>::v_chunk(base, c), fb, p.layout,
                           c * C::kChunkElemsV, hk, j * kBN, it.b, pol_kv);
              }
            }
          }
        }
        if (!ok) break;
        if constexpr (kDynamic) {
          // The next item: a CTA of this grid that has not started, if any.
          ptx::mbar_arrive_expect_tx(bar(B::kClc), 16);
          ptx::clc_try_cancel(sm.clc_resp, bar(B::kClc));
          clc_pending = true;
          ok = ptx::mbar_wait(bar(B::kClc), clc_par, abort, status, 1);
          if (!ok) break;
          clc_pending = false;
          clc_par ^= 1u;
          int x = 0;
          more = ptx::clc_query(sm.clc_resp, x);
          w = x;
        } else {
          w = item_index(r + 1, blockIdx.x, gridDim.x);
          more = w < p.total_items;
        }
      }
      if (!ok) {
        if (clc_pending) ptx::mbar_drain(bar(B::kClc), clc_par);
        // Unwind: let every copy this thread issued land before the CTA's
        // shared memory is released (each copy completes on the last
        // arming of some full barrier).
        for (int x = 0; x < NS; ++x)
          if ((armed >> x) & 1u) ptx::mbar_drain(bar(B::kSlotFull + x), ((fpar >> x) & 1u) ^ 1u);
        for (int s = 0; s < 2; ++s)
          if ((q_used >> s) & 1u) ptx::mbar_drain(bar(B::kQFull + s), ((q_par >> s) & 1u) ^ 1u);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs the issuing loop (every value in it is
    // warp-uniform) and one elected lane issues each MMA and commit.
    {
      uint32_t q_par = 0, pv_par = 0;  // bit s: phase parity per stage
      uint32_t p_count[2] = {0u, 0u};             // P tiles received per stage
      uint32_t t = 0;     // slot ring: K/V tiles consumed so far
      Ring<C> ring;       // chunk-piece ring: placement
      uint32_t fpar = 0;  // bit x: phase parity of full barrier x to wait for next
      bool ok = true;
      // Base descriptors; an MMA adds its byte offset >> 4 to the start
      // address field (addresses stay below 256 KB, so no carry leaves it).
      const uint64_t dq0 = ptx::smem_desc(q_smem, 16, 8 * C::kSwzQK, C::kSwzModeQK);
      const uint64_t dk0 = ptx::smem_desc(slots_smem, 16, 8 * C::kSwzQK, C::kSwzModeQK);
      const uint64_t dv0 = ptx::smem_desc(slots_smem, C::kChunkBytesV, 1024, 2u);

      // S_s = Q_s K^T, K in slot `kb` (slot ring) or with chunk 0 in piece
      // `kb` (chunk-piece ring).
      auto issue_s = [&](int s, uint32_t kb) {
        const uint64_t dq = dq0 + ((s * C::kTileBytesQK) >> 4);
        const uint32_t d_tmem = tmem + s * 128;
        if constexpr (!C::kChunkPieces) {
          const uint64_t dk = dk0 + ((kb * C::kSlotBytes) >> 4);
#pragma unroll
          for (int c = 0; c < C::kChunksQK; ++c) {
#pragma unroll
            for (int kk = 0; kk < C::kSwzQK / 32; ++kk) {
              const uint32_t off = (c * C::kChunkBytesQK + kk * 32) >> 4;
              ptx::mma_ss_elect<C::kF8>(d_tmem, dq + off, dk + off, C::kIdescQK, (c | kk) != 0);
            }
          }
        } else {
          // Not unrolled over chunks: the smaller issuer code measured up to
          // 17 % faster on the BF16 d_qk = 192 form (same MMAs, same order).
#pragma unroll 1
          for (int c = 0; c < C::kChunksQK; ++c) {
            const uint64_t dk = dk0 + (Ring<C>::k_chunk(kb, c) >> 4);
#pragma unroll
            for (int kk = 0; kk < C::kSwzQK / 32; ++kk) {
              const uint32_t qoff = (c * C::kChunkBytesQK + kk * 32) >> 4;
              const uint32_t koff = (kk * 32) >> 4;
              ptx::mma_ss_elect<C::kF8>(d_tmem, dq + qoff, dk + koff, C::kIdescQK, (c | kk) != 0);
            }
          }
        }
      };
      // O_s (+)= P V, V with chunk 0 in ring piece `vb` (its chunks are
      // kChunkBytesV apart, the descriptor's leading offset), and P read from
      // tensor memory at column offset p_col of S_s (FP8 keeps a residual P
      // term at 32).
      auto issue_pv = [&](int s, uint32_t vb, bool acc_first, uint32_t p_col) {
        const uint64_t dv = dv0 + (Ring<C>::v_chunk(vb, 0) >> 4);
        const uint32_t a_tmem = tmem + s * 128 + p_col;
        const uint32_t d_tmem = tmem + 256 + s * 128;
        if constexpr (C::kBlockScale) {
          // Slice ks of P (keys 32 ks .. 32 ks + 31) with its scale factors.
          const uint32_t sfa = tmem + s * 128 + kSfaCol, sfb = tmem + s * 128 + kSfbCol;
#pragma unroll
          for (int ks = 0; ks < kBN / C::kUmmaK; ++ks)
            ptx::mma_ts_bs_elect(d_tmem, a_tmem + ks * 8, dv + ((ks * C::kUmmaK * 128) >> 4),
                                 C::idesc_pv_bs(ks), sfa, sfb, (acc_first || ks > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int ks = 0; ks < kBN / C::kUmmaK; ++ks)
            ptx::mma_ts_elect<C::kF8>(d_tmem, a_tmem + ks * 8,
                                      dv + ((ks * C::kUmmaK * 128) >> 4), C::kIdescPV,
                                      (acc_first || ks > 0) ? 1u : 0u);
        }
      };

      for (int r = 0; ok; ++r) {
        int w = -1;
        ok = take_item(r, w);
        if (!ok || w < 0) break;
        const Item it = decode_item(w, p);
        const int nst = it.n1 > 0 ? 2 : 1;
        for (int s = 0; s < nst && ok; ++s) {
          ok = warp_wait(bar(B::kQFull + s), (q_par >> s) & 1u, abort, status, lane);
          q_par ^= 1u << s;
        }
        if (!ok) break;
        // Prologue: S of K/V tile 0 for both stages.
        uint32_t kb = 0, kl = 0, slot_k;
        if constexpr (!C::kChunkPieces) {
          slot_k = t % NS;
          ++t;
          kb = slot_k;
        } else {
          slot_k = ring.place(false, kb, kl);
        }
        ok = warp_wait(bar(B::kSlotFull + slot_k), (fpar >> slot_k) & 1u, abort, status, lane);
        if (!ok) break;
        fpar ^= 1u << slot_k;
        ptx::tc_fence_after();
        issue_s(0, kb);
        ptx::mma_commit_elect(bar(B::kSFull + 0));
        if (it.n1 > 0) {
          issue_s(1, kb);
          ptx::mma_commit_elect(bar(B::kSFull + 1));
        }
        ptx::mma_commit_elect(bar(B::kSlotEmpty + slot_k));

        for (int j = 0; j < it.nload && ok; ++j) {
          // Slot ring: one wait covers V_j and (when there is a next tile)
          // K_j+1.
          uint32_t vb = 0, vl = 0, slot_v;
          if constexpr (!C::kChunkPieces) {
            slot_v = t % NS;
            ++t;
            vb = slot_v;
          } else {
            slot_v = ring.place(true, vb, vl);
          }
          const bool has_next = j + 1 < it.nload;
          if (has_next) {
            if constexpr (!C::kChunkPieces) {
              slot_k = t % NS;
              ++t;
              kb = slot_k;
            } else {
              slot_k = ring.place(false, kb, kl);
            }
          }
          ok = warp_wait(bar(B::kSlotFull + slot_v), (fpar >> slot_v) & 1u, abort, status, lane);
          if (!ok) break;
          fpar ^= 1u << slot_v;
          // Chunk-piece ring: K_j+1 has its own full barrier, waited for
          // before its first S; V_j is released right after its last P V
          // (stage 1 when it runs this step), so the pieces it frees start
          // loading while the last S of the step runs.
          if constexpr (C::kRollStages) {
            bool k_pending = C::kChunkPieces && has_next;
            const int s_last_v = j < it.n1 ? 1 : 0;
            // One stage's P V and next S.  Returns false when a wait gave up.
            auto run_stage = [&](int s) -> bool {
              const int ns = s == 0 ? it.n0 : it.n1;
              if (j >= ns) return true;
              // P of stage s: named barrier 1 + s with its four softmax warps.
              ptx::bar_sync(1 + s, 160);
              // The abort flag and the lo-term flag are loaded here and used
              // only once the P V MMAs are issued: a shared-memory load from
              // this thread takes hundreds of cycles while the tensor core
              // streams its operands, and the MMA queue would run dry if the
              // issue waited for it.  (Should a softmax warp have given up,
              // the P V MMAs read a P that nobody wrote: every operand is in
              // range, and the launch's results are void anyway.)
              const int abort_raw = *abort;
              uint32_t lo_raw = 0;
              if constexpr (C::kF8) lo_raw = sm.pflag[s];
              const uint32_t pcount = s == 0 ? ++p_count[0] : ++p_count[1];
              ptx::tc_fence_after();
              issue_pv(s, vb, j > 0, 0);
              if (C::kF8 && __shfl_sync(0xffffffffu, lo_raw, 0) == pcount)
                issue_pv(s, vb, true, 32);  // lo term
              if (__shfl_sync(0xffffffffu, abort_raw, 0)) {
                ok = false;
                return false;
              }
              if constexpr (C::kChunkPieces) {
                if (s == s_last_v) ptx::mma_commit_elect(bar(B::kSlotEmpty + slot_v));
              }
              if (p.serialize_pv && j + 1 < ns) {
                // Verification mode: P (aliasing S) is fully consumed before the
                // next S MMA of this stage overwrites it.
                ptx::mma_commit_elect(bar(B::kPvDone + s));
                ok = warp_wait(bar(B::kPvDone + s), (pv_par >> s) & 1u, abort, status, lane);
                pv_par ^= 1u << s;
                if (!ok) return false;
              }
              if (j + 1 < ns) {
                if constexpr (C::kChunkPieces) {
                  if (k_pending) {
                    ok = warp_wait(bar(B::kSlotFull + slot_k), (fpar >> slot_k) & 1u, abort,
                                        status, lane);
                    if (!ok) return false;
                    fpar ^= 1u << slot_k;
                    k_pending = false;
                    ptx::tc_fence_after();
                  }
                }
                issue_s(s, kb);
                ptx::mma_commit_elect(bar(B::kSFull + s));
              } else {
                ptx::mma_commit_elect(bar(B::kOFull + s));
              }
              return true;
            };
#pragma unroll 1
            for (int s = 0; s < 2 && ok; ++s) ok = run_stage(s);
          } else {
            // BF16 d_qk = 128 (whole-tile slots): the same steps, unrolled
            // over the two stages.
            for (int s = 0; s < 2; ++s) {
              const int ns = s == 0 ? it.n0 : it.n1;
              if (j >= ns) continue;
              ptx::bar_sync(1 + s, 160);
              const int abort_raw = *abort;   // used after the P V MMAs (as above)
              ++p_count[s];
              ptx::tc_fence_after();
              issue_pv(s, vb, j > 0, 0);
              if (__shfl_sync(0xffffffffu, abort_raw, 0)) {
                ok = false;
                break;
              }
              if (p.serialize_pv && j + 1 < ns) {
                ptx::mma_commit_elect(bar(B::kPvDone + s));
                ok = warp_wait(bar(B::kPvDone + s), (pv_par >> s) & 1u, abort, status, lane);
                pv_par ^= 1u << s;
                if (!ok) break;
              }
              if (j + 1 < ns) {
                issue_s(s, kb);
                ptx::mma_commit_elect(bar(B::kSFull + s));
              } else {
                ptx::mma_commit_elect(bar(B::kOFull + s));
              }
            }
          }
          if (!ok) break;
          if constexpr (!C::kChunkPieces) ptx::mma_commit_elect(bar(B::kSlotEmpty + slot_v));
          if (has_next) ptx::mma_commit_elect(bar(B::kSlotEmpty + slot_k));
        }
        if (!ok) break;
        for (int s = 0; s < nst; ++s) ptx::mma_commit_elect(bar(B::kQEmpty + s));
      }
      // Every MMA this thread issued completes before tensor memory is freed.
      ptx::mma_commit_elect(bar(B::kDrain));
      ptx::mbar_drain(bar(B::kDrain), 0);
    }
    __syncwarp();
  }
  } else {
    ptx::setmaxnreg_inc<C::kSoftmaxRegs>();
    // ------------------------------------------------------------- softmax
    const int s = warp >> 2;            // stage
    const int wq = warp & 3;            // lane quarter of TMEM this warp may access
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + (s ? 128u : 0u);
    const uint32_t t_o = tmem + lane_base + (s ? 384u : 256u);
    float c_log2 = p.softmax_scale * 1.4426950408889634f;
    float o_extra = 1.0f;
    if constexpr (C::kF8) {
      c_log2 *= __ldg(p.q_descale) * __ldg(p.k_descale);
      o_extra = __ldg(p.v_descale);
    }
    uint32_t s_uses = 0, o_uses = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      int w = -1;
      ok = take_item(r, w);
      if (!ok || w < 0) break;
      const Item it = decode_item(w, p);
      const int ns = s == 0 ? it.n0 : it.n1;
      if (ns == 0) continue;
      const int tile = 2 * it.u + s;
      float m_ref = -INFINITY;  // reference maximum, base-2 units of the scaled score
      float l = 0.f;            // sum of 2^(x - m_ref + kPLog2Scale), unrounded (for LSE)
      float lr = 0.f;           // the same sum over the rounded (BF16 / e4m3) values that
                                // multiply V: the denominator of O
      for (int j = 0; j < ns; ++j) {
        ok = warp_wait(bar(B::kSFull + s), s_uses & 1u, abort, status, lane);
        if (!ok) break;
        ++s_uses;
        ptx::tc_fence_after();
        // S row: columns 0..31 are loaded and waited for; 32..127 are
        // requested at once and waited for after the first 32 exp2 (a
        // tensor-memory load takes hundreds of cycles while the tensor core
        // streams, so the wait covers as few columns as possible).
        uint32_t v[128];
        ptx::tmem_ld32_wait(t_s, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        ptx::tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        ptx::tmem_ld64_nowait(t_s + 64, *reinterpret_cast<uint32_t(*)[64]>(&v[64]));
        auto wait_rest = [&]() {
          ptx::tmem_wait_ld_dep32(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          ptx::tmem_wait_ld_dep64(*reinterpret_cast<uint32_t(*)[64]>(&v[64]));
        };
        float* f = reinterpret_cast<float*>(v);
        const bool diag = j == tile;
        if (diag) {
          // Diagonal tile: key column c is in the future of the row when
          // c exceeds the row's index in the tile.
          wait_rest();
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > row_in_tile) f[c] = -INFINITY;
        }
        // Accuracy of the rounded P (decided per warp from the tile's actual
        // maximum): a probability that carries at least 1/8 (BF16) or 1/16
        // (FP8; 1/32 with the rounded-P denominator) of the row's mass so far
        // would show its rounding in the
        // normalised output.  BF16 then sums the denominator over the same
        // rounded values that multiply V (ZYFA README, "Accuracy"); FP8
        // keeps P as two e4m3 terms, hi + lo, lo being the rounding residual
        // of hi (about 8 significant bits together; always on a row's first
        // tile), and the MMA issuer adds a second
        // P V product for lo when any warp of the stage flags the tile (the
        // other warps store zeros as their lo term).  On other tiles the
        // rounding errors average out and the unrounded sum stands in.
        float rs = 0.f, rr = 0.f;
        bool exact = false, two_term = false;
        if constexpr (C::kBlockScale) {
          // Per-slice scales need each slice's maximum before its exp2, so
          // the tile maximum is known first and a rescale of O, when the
          // maximum passes the reference by more than tau, precedes P (no
          // recomputation).  Two-term P as below: on the first tile, the
          // diagonal tile, a rescaled tile, and where one probability
          // carries at least 1/32 of the row's mass.
          float xm[4];
          xm[0] = row_max32(f);
          wait_rest();
          xm[1] = row_max32(f + 32);
          xm[2] = row_max32(f + 64);
          xm[3] = row_max32(f + 96);
          const float mx = fmaxf(fmaxf(xm[0], xm[1]), fmaxf(xm[2], xm[3])) * c_log2;
          bool any_need = false;
          if (j == 0) {
            m_ref = mx;
          } else {
            const bool need = mx > m_ref + C::kTau;
            any_need = __any_sync(0xffffffffu, need);
            if (any_need) {
              const float alpha = need ? ptx::ex2(m_ref - mx) : 1.0f;
              if (need) {
                l *= alpha;
                lr *= alpha;
                m_ref = mx;
              }
              rescale_o(t_o, alpha);
            }
          }
          const float neg_m = C::kPLog2Scale - m_ref;
          float ex[4];
          uint32_t sfw = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ex[k] = slice_exponent(xm[k], c_log2, m_ref);
            sfw |= static_cast<uint32_t>(127 - static_cast<int>(ex[k])) << (8 * k);
          }
          const uint32_t unit[4] = {0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu};
          ptx::tmem_st1(t_s + kSfaCol + wq, sfw);
          ptx::tmem_st4(t_s + kSfbCol, unit);
          if (j == 0 || diag || any_need) {
            two_term = true;
            if (lane == 0) sm.pflag[s] = s_uses;
            produce_bs<C, true, true>(f, c_log2, neg_m, ex, t_s, rs, rr);
          } else {
            produce_bs<C, true, false>(f, c_log2, neg_m, ex, t_s, rs, rr);
            const float p_max = ptx::ex2(mx + neg_m);
            two_term = __any_sync(0xffffffffu, p_max * C::kAccRatio > l + rs);
            if (two_term) {
              if (lane == 0) sm.pflag[s] = s_uses;
              produce_bs<C, false, true>(f, c_log2, neg_m, ex, t_s, rs, rr);
            }
          }
        } else if (j == 0) {
          // First tile of the row: the reference is this tile's maximum.
          wait_rest();
          m_ref = row_max128(f) * c_log2;
          exact = !C::kF8;
          two_term = C::kF8;
          if (C::kF8 && lane == 0) sm.pflag[s] = s_uses;
          produce_tile<C, !C::kF8>(f, c_log2, C::kPLog2Scale - m_ref, t_s, two_term, rs, rr);
        } else {
          // Exp2 against the current reference while the tile maximum is
          // formed; a tile whose maximum passes the reference by more than
          // tau is recomputed after the rescale (rare: tau is large).
          float neg_m = C::kPLog2Scale - m_ref;
          float2 sacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          // FP8: the tests run on the packed P (threshold_addend): a code at
          // or above that of min(kPCap, l / kAccRatio) sends the warp to the
          // exact path.  Both tests are then conservative: p > kPCap or
          // p * kAccRatio > l + rs implies such a code (rounding to e4m3 is
          // monotonic and l <= l + rs).
          uint32_t tk = 0, tacc = 0;
          if constexpr (C::kF8) {
            const uint32_t cap_code = ptx::pack_e4m3x4(C::kPCap, 0.f, 0.f, 0.f) & 0xFFu;
            const uint32_t acc_code = ptx::pack_e4m3x4(l * (1.0f / C::kAccRatio), 0.f, 0.f, 0.f) & 0xFFu;
            tk = threshold_addend(acc_code < cap_code ? acc_code : cap_code);
          }
          // BF16 d_qk = 128: per 32-key chunk sums, the largest of which
          // bounds every p of the tile (the whole tile sum elsewhere).
          float cs[4];
          float* csp = C::kChunkBound ? cs : nullptr;
          produce_half<C, false, C::kF8>(f, c_log2, neg_m, t_s, 0, false, sacc, rr, tk, &tacc, 0, 1, csp);
          wait_rest();
          produce_half<C, false, C::kF8>(f, c_log2, neg_m, t_s, 0, false, sacc, rr, tk, &tacc, 1, 1, csp);
          produce_half<C, false, C::kF8>(f, c_log2, neg_m, t_s, 1, false, sacc, rr, tk, &tacc, 0, 2, csp);
          if constexpr (!C::kChunkBound) {
            const float2 t2 = __fadd2_rn(sacc[0], sacc[1]);
            rs = t2.x + t2.y;
          } else {
            rs = (cs[0] + cs[1]) + (cs[2] + cs[3]);
          }
          // The unrounded sum bounds every p of the tile (all p >= 0).  When
          // it is small enough, neither the rescale test nor the accuracy
          // test can fire and the tile maximum is not needed (the 0.1%
          // margin covers the rounding of exp2 and of the sum); otherwise
          // the warp forms the maximum and takes the tests exactly.
          const float bound =
              (C::kChunkBound ? fmaxf(fmaxf(cs[0], cs[1]), fmaxf(cs[2], cs[3])) : rs) * 1.001f;
          // (BF16 with the rounded-P denominator on every tile has no
          // accuracy test: the denominator it would switch to is already
          // the one in use; only the rescale test remains.)
          const bool quiet = C::kF8 ? (tacc & 0x80808080u) == 0u
                                    : (bound <= C::kPCap &&
                                       (C::kRoundedP || bound * C::kAccRatio <= l + rs));
          if ((!C::kF8 && diag) || !__all_sync(0xffffffffu, quiet)) {
          const float mx = row_max128(f) * c_log2;
          const bool need = mx > m_ref + C::kTau;
          const bool any_need = __any_sync(0xffffffffu, need);
          if (any_need) {
            const float alpha = need ? ptx::ex2(m_ref - mx) : 1.0f;
            if (need) {
              l *= alpha;
              lr *= alpha;
              m_ref = mx;
            }
            rescale_o(t_o, alpha);
            // P of this tile is computed again below (redo_*) against the
            // moved reference, exactly the values a non-speculative pass
            // would have produced, once the speculative stores to the same
            // columns have completed.
            ptx::tmem_wait_st();
            neg_m = C::kPLog2Scale - m_ref;
          }
          const float p_max = ptx::ex2(mx + neg_m);   // largest p of the tile (x pre-scale)
          if constexpr (C::kF8) {
            // A recomputed tile takes the two-term P in the same exp2 pass
            // (right after a rescale its maximum carries most of the mass
            // the row has seen, so the test below would pass anyway).
            two_term = any_need || __any_sync(0xffffffffu, p_max * C::kAccRatio > l + rs);
            if (two_term) {
              if (lane == 0) sm.pflag[s] = s_uses;
              redo_fp8<C>(f, c_log2, neg_m, t_s, any_need, rs, rr);
            }
          } else {
            // A recomputed tile takes the rounded-sum denominator in the same
            // exp2 pass (right after a rescale its maximum carries most of
            // the mass the row has seen, so the test would pass anyway).
            exact = any_need ||
                    (!C::kRoundedP && __any_sync(0xffffffffu, p_max * 8.0f > l + rs));
            if (exact) redo_bf16(f, c_log2, neg_m, t_s, any_need, rs, rr);
          }
          }
        }
        // FP8: a two-term tile's lane 0 has stored the tile's count as the
        // lo-term flag as soon as the decision was taken (the store then
        // completes during the lo pass, not at the fence below); other tiles
        // store zeros as their lo term.  The MMA issuer reads the flag of
        // this tile only after the arrival below, and its read of the
        // previous tile's flag returned before it issued this tile's S, so
        // the early store overwrites nothing it still needs.
        if (C::kF8 && !two_term) {
          const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
          for (int c = 0; c < 4; ++c) ptx::tmem_st8(t_s + 32 + c * 8, z);
        }
        l += rs;
        lr += (exact || C::kRoundedP) ? rr : rs;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        // P ready: the four softmax warps of the stage arrive on hardware
        // barrier 1 + s, on which the MMA issuer warp waits (bar.sync).  A
        // hardware barrier wakes the issuer sooner than an mbarrier phase
        // (1-3 %).  It has no time limit, so its arrivals are guaranteed by
        // construction: every wait a softmax warp passes before an arrival
        // is bounded, a warp that gives up arrives once more on its way out
        // (below), and the issuer reads the abort flag after every wait
        // (testing it once that stage's P V MMAs are issued).  Lane 0's
        // lo-term flag store, on two-term FP8 tiles only, is fenced before
        // the arrival; other tiles store nothing the issuer reads.
        if (C::kF8 && two_term && lane == 0) __threadfence_block();
        __syncwarp();
        ptx::bar_arrive(1 + s, 160);
      }
      if (!ok) break;
      // Epilogue: O * v_descale / lr as BF16 (FP8: the 2^2 pre-scale of P
      // cancels, lr summing the same pre-scaled values), and the LSE.
      ok = warp_wait(bar(B::kOFull + s), o_uses & 1u, abort, status, lane);
      if (!ok) break;
      ++o_uses;
      ptx::tc_fence_after();
      const int row = tile * kBM + row_in_tile;
      const bool valid = row < p.S;
      const float inv = o_extra / lr;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
      const int64_t orow =
          p.layout == 0
              ? ((static_cast<int64_t>(it.b) * p.S + row) * p.H + it.h) * kDV
              : ((static_cast<int64_t>(it.b) * p.H + it.h) * p.S + row) * kDV;
      // All of O in one tensor-memory load and wait (each load waits
      // hundreds of cycles while the other stage's MMAs stream).
      uint32_t o[128];
      ptx::tmem_ld128_wait(t_o, o);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack_bf16x2(__uint_as_float(o[32 * c + 2 * i]) * inv,
                                   __uint_as_float(o[32 * c + 2 * i + 1]) * inv);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (valid && p.lse != nullptr) {
        // Mode 2 takes the LSE from the same rounded sum as the
        // denominator (results over different key ranges then merge
        // consistently; ZYFA README, "Accuracy").
        const float lsum = (C::kRoundedP && p.rounded_p == 2) ? lr : l;
        p.lse[(static_cast<int64_t>(it.b) * p.H + it.h) * p.S + row] =
            (m_ref + log2f(lsum) - C::kPLog2Scale) * 0.6931471805599453f;
      }
      ptx::tc_fence_before();
    }
    // A softmax warp that gives up releases an MMA issuer that may be waiting
    // for its P (the issuer then sees the abort flag and unwinds).
    if (!ok) ptx::bar_arrive(1 + s, 160);
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------- host side

// The dynamic shared-memory limit is raised once per device and
// instantiation.  Should a launch still be refused (the attribute is lost
// when a device is reset), it is raised again and the launch retried once.
template <int DT, int DQK, int RP, int BS = 0, int DS = 0>
static int launch_one(const FwdParams& p, const TensorMaps& m, int grid, int device,
                      cudaStream_t stream) {
  using C = Cfg<DT, DQK, RP, BS>;
  static std::atomic<uint64_t> attr_set{0};   // bit d: raised on device d
  auto kern = zyfa_fwd_kernel<DT, DQK, RP, BS, DS>;
  const uint64_t bit = 1ull << device;
  auto raise_limit = [&]() -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e == cudaSuccess) attr_set.fetch_or(bit, std::memory_order_relaxed);
    return e;
  };
  if (!(attr_set.load(std::memory_order_relaxed) & bit)) {
    const cudaError_t e = raise_limit();
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(m.q, m.k, m.v, p);
  cudaError_t e = cudaGetLastError();
  if (e == cudaErrorInvalidValue || e == cudaErrorLaunchOutOfResources) {
    if ((e = raise_limit()) != cudaSuccess) return e;
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(m.q, m.k, m.v, p);
    e = cudaGetLastError();
  }
  return e;
}

int launch_fwd(int dtype, int d_qk, const FwdParams& p, const TensorMaps& maps, int grid,
               int device, cudaStream_t stream) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  if (p.dynamic_schedule) {
    // Dynamic schedule: the default softmax modes only (the host sizes the
    // grid for the schedule it asks for, see api.cpp).
    if (dtype == 0 && d_qk == 128) return launch_one<0, 128, 0, 0, 1>(p, maps, grid, device, stream);
    if (dtype == 0 && d_qk == 192) return launch_one<0, 192, 0, 0, 1>(p, maps, grid, device, stream);
    if (dtype == 1 && d_qk == 128) return launch_one<1, 128, 0, 0, 1>(p, maps, grid, device, stream);
    if (dtype == 1 && d_qk == 192) return launch_one<1, 192, 0, 0, 1>(p, maps, grid, device, stream);
    return cudaErrorInvalidValue;
  }
  if (dtype == 1 && p.block_scale) {
    if (p.rounded_p == 0) {
      if (d_qk == 128) return launch_one<1, 128, 0, 1>(p, maps, grid, device, stream);
      if (d_qk == 192) return launch_one<1, 192, 0, 1>(p, maps, grid, device, stream);
    } else {
      if (d_qk == 128) return launch_one<1, 128, 1, 1>(p, maps, grid, device, stream);
      if (d_qk == 192) return launch_one<1, 192, 1, 1>(p, maps, grid, device, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (p.rounded_p == 0) {
    if (dtype == 0 && d_qk == 128) return launch_one<0, 128, 0>(p, maps, grid, device, stream);
    if (dtype == 0 && d_qk == 192) return launch_one<0, 192, 0>(p, maps, grid, device, stream);
    if (dtype == 1 && d_qk == 128) return launch_one<1, 128, 0>(p, maps, grid, device, stream);
    if (dtype == 1 && d_qk == 192) return launch_one<1, 192, 0>(p, maps, grid, device, stream);
  } else {
    if (dtype == 0 && d_qk == 128) return launch_one<0, 128, 1>(p, maps, grid, device, stream);
    if (dtype == 0 && d_qk == 192) return launch_one<0, 192, 1>(p, maps, grid, device, stream);
    if (dtype == 1 && d_qk == 128) return launch_one<1, 128, 1>(p, maps, grid, device, stream);
    if (dtype == 1 && d_qk == 192) return launch_one<1, 192, 1>(p, maps, grid, device, stream);
  }
  return cudaErrorInvalidValue;
}

template <int DT, int DQK>
static void geometry_of(KernelGeometry* g) {
  using C = Cfg<DT, DQK>;
  g->smem_bytes = C::kSmemBytes;
  g->qk_box_elems = C::kChunkElemsQK;
  g->qk_swizzle = C::kSwzQK;
  g->v_box_elems = C::kChunkElemsV;
  g->num_slots = C::kNumPieces;
}

int kernel_geometry(int dtype, int d_qk, KernelGeometry* g) {
  if (dtype == 0 && d_qk == 128) return geometry_of<0, 128>(g), 0;
  if (dtype == 0 && d_qk == 192) return geometry_of<0, 192>(g), 0;
  if (dtype == 1 && d_qk == 128) return geometry_of<1, 128>(g), 0;
  if (dtype == 1 && d_qk == 192) return geometry_of<1, 192>(g), 0;
  return -1;
}

int read_device_status(int* value, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_zyfa_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (reset) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_zyfa_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace zyfa
