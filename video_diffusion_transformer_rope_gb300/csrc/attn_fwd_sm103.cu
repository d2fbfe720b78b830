// Warp-specialised flash-attention forward with 3D RoPE for sm_103a (GB300), plus the
// Q/K-rotation prepass it can stream from.
//
// Operation: vidax: A Unified JAX Framework for Video Generative Models on Accelerator
// Meshes, §2 "3D RoPE, 3D VAEs, and flash attention" (rotary 3D positions on Q and K, then
// attention without materialising the N x N scores).  bf16 in/out, d = 128, fp32 softmax
// statistics and accumulators.  The rotated Q and K are rounded to fp16 (11-bit significand,
// 8x finer than bf16) for the QK^T product; P and V enter the PV product as bf16.
//
// One CTA owns 256 query rows (two 128-row Q tiles) of one (batch, head) and streams every
// 128-key K/V tile of that head (or, with a block mask, the tiles its mask row selects).
// Warp roles (one warpgroup each, registers rebalanced with setmaxnreg once the roles split):
//
//   WG0  warps 0-3   softmax + epilogue for Q tile 0 (thread = query row = TMEM lane)
//   WG1  warps 4-7   softmax + epilogue for Q tile 1
//   WG2  warps 8-11  RoPE: rotate the Q tiles in shared memory as they land (bf16 -> fp16,
//                    in place) unless the prepass already did, or gather + rotate a query
//                    subset straight from global memory; in the fused-K mode also every K tile
//   WG3  warp 12     TMA producer: Q tiles once, then K/V tiles through the rings
//        warp 13     tcgen05 MMA issuer (the whole warp runs the loop, one elected lane
//                    issues) and TMEM owner (in a CTA pair: rank 0 only)
//        warp 14     rank 1 of a CTA pair: relays its landed Q/K/V halves to rank 0 (V only
//                    with the fused K rotation, where rank 1's WG2 signals its rotated tiles)
//        warp 15     idle
//
// K modes.  Prepass (default): a separate kernel rotates K once per token into an fp16
// workspace and the attention kernel streams that, so no K rotation sits in the hot loop.
// The prepass rotates (and scales) Q as well and the Q tiles arrive ready through TMA; only a
// query subset (gathered rows), the fused-K mode and the no-allocation entry have WG2 rotate
// each CTA's Q tiles.
// Fused: TMA brings raw bf16 K and WG2 rotates each K tile in shared memory before the MMA
// reads it (every CTA of a head repeats this for every K tile).  On CTA pairs (the default for
// fused calls) each CTA rotates only its own 64 keys of every K tile, with cosines and sines
// from the special-function unit (no table in shared memory), and rank 1's WG2 signals the
// rotated half to rank 0, whose MMA warp waits for both halves before it issues.
// Split (precise): as prepass, but every rotated Q/K value x is kept as two fp16 numbers,
// hi = fp16(x) and lo = fp16(x - hi), and S = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T (about 22
// significant bits per operand instead of 11) for inputs whose logits reach the hundreds.
// Three QK products and one-stage K/V rings (shared memory holds Q hi+lo and K hi+lo); run by
// CTA pairs (below), each CTA holds half of every K/V tile and its rings hold two stages.
//
// CTA pairs (long dense sequences): two CTAs of a cluster take consecutive query blocks of one
// (b, h).  Each loads only half of every K tile (keys 0-63 or 64-127) and half of every V tile
// (channels 0-63 or 64-127) into its own 4-stage rings, and the rank-0 CTA issues cta_group::2
// MMAs (M = 256: both CTAs' Q tiles, N = 128 read from both CTAs' halves) that write each
// CTA's rows into its own tensor memory; the multicast commits tell both CTAs.  Rank 1 relays
// "my half has landed" and "my P is stored" to rank 0 with remote mbarrier arrivals.  Same
// softmax and epilogue per CTA; half the shared-memory operand reads and L2->SM traffic.
//
// TMEM (512 columns x 128 lanes, fp32): S0 [0,128)  S1 [128,256)  O0 [256,384)  O1 [384,512).
// P_i (bf16, two per column) overwrites the first 64 columns of S_i and is the A operand of
// the PV MMA straight from TMEM.  MMA issue order per key tile j:
//     S0(j) = Q0 K_j^T ;  O1 += P1(j-1) V_{j-1} ;  S1(j) = Q1 K_j^T ;  O0 += P0(j) V_j
// so softmax of one Q tile overlaps the tensor-core work of the other.  Completion of S_i(j)
// implies completion of every earlier MMA, so O_i may be rescaled as soon as S_i(j) is seen.
// The online softmax works in the log2 domain: the rotated Q tiles are stored already
// multiplied by scale*log2(e), so S comes out of the MMA in log2 units and p = 2^(s - m).
// Each tile's exponentials are taken against the running maximum m and kept when the row
// sum shows every p <= 256; only otherwise (the first tile, or scores that rose) is the tile
// maximum computed, m moved there, l and O rescaled and the row redone.
//
// Epilogue: each softmax warpgroup writes O/l (bf16) into its Q tile buffer, free once the
// last MMA has completed, in the same swizzled layout, and one thread stores the tile with
// TMA (a query subset scatters its rows with plain stores instead).
//
// Shared memory: Q 2x32 KB, K ring, V ring (32 KB per stage), each tile stored as two
// 128-row x 128-byte halves in the 128-byte-swizzled layout TMA writes; then (fused mode,
// when it fits) the cos/sin table, then the mbarriers.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cmath>

#include "sm103_ptx.cuh"
#include "vdx_internal.h"

namespace vdx {
namespace {

constexpr int kBM = 128;                 // rows per Q tile
constexpr int kQTiles = 2;               // Q tiles per CTA
constexpr int kRowsPerCta = kBM * kQTiles;
constexpr int kBN = 128;                 // keys per K/V tile
constexpr int kD = 128;
constexpr int kTileBytes = kBN * kD * 2; // 32 KB
constexpr int kHalfBytes = kTileBytes / 2;
constexpr int kThreads = 512;
constexpr int kTmemCols = 512;
constexpr int kMaxStages = 4;
constexpr int kMaxDynSmem = 232448;      // sm_100-family opt-in limit per CTA


// kModePair: the prepass mode run by a cluster of two CTAs (a CTA pair) that share every
// K/V tile: each CTA holds half of it (keys 0-63 or 64-127 of a K tile, channels 0-63 or
// 64-127 of a V tile) and the pair's rank-0 CTA issues cta_group::2 MMAs over both CTAs' 256
// query rows.
// kModePairSplit: the split mode run by CTA pairs (each CTA: Q hi + lo, 2-stage rings of K
// halves hi + lo and V halves).
// kModePairFused: the fused-K mode run by CTA pairs: each CTA rotates its own two Q tiles and
// its half (64 keys) of every K tile in shared memory, so the per-CTA rotation work is half
// that of kModeFused.
enum : int {
  kModePrepass = 0, kModeFused = 1, kModeSplit = 2, kModePair = 3, kModePairSplit = 4, kModePairFused = 5
};

template <int kMode>
struct Layout {
  static constexpr bool kFusedK = kMode == kModeFused || kMode == kModePairFused;
  static constexpr bool kSplit = kMode == kModeSplit || kMode == kModePairSplit;
  static constexpr bool kPair = kMode == kModePair || kMode == kModePairSplit || kMode == kModePairFused;
  static constexpr int kKStages =
      kMode == kModePrepass ? 3
      : (kMode == kModeFused ? 2 : ((kMode == kModePair || kMode == kModePairFused) ? 4 : (kMode == kModePairSplit ? 2 : 1)));
  static constexpr int kVStages =
      kMode == kModeSplit ? 1 : ((kMode == kModePair || kMode == kModePairFused) ? 4 : 2);
  // K stage: one tile (hi), or hi + lo; a CTA pair holds half of each
  static constexpr int kKStageBytes = (kSplit ? 2 * kTileBytes : kTileBytes) / (kPair ? 2 : 1);
  static constexpr int kVStageBytes = kPair ? kTileBytes / 2 : kTileBytes;
  static constexpr int kOffQ = 0;                                              // Q (hi) tiles
  static constexpr int kOffQlo = kOffQ + kQTiles * kTileBytes;                 // Q lo tiles
  static constexpr int kOffK = kOffQlo + (kSplit ? kQTiles * kTileBytes : 0);
  static constexpr int kOffV = kOffK + kKStages * kKStageBytes;
  static constexpr int kOffTab = kOffV + kVStages * kVStageBytes;
  // Registers per thread after the role split (sum over the 4 warpgroups = 512 x 128 at
  // launch); the split mode's MMA warp issues three QK chains and needs more.
  static constexpr uint32_t kRegsSoftmax = kSplit ? 160 : 184;
  static constexpr uint32_t kRegsRope = kSplit ? 64 : 72;
  static constexpr uint32_t kRegsCtl = kSplit ? 128 : 72;
  static_assert(2 * kRegsSoftmax + kRegsRope + kRegsCtl <= 4 * 128, "register split over budget");
};

// Wait sites recorded in the error word when a bounded wait gives up.
enum : int {
  kSiteQFull = 1, kSiteKFull, kSiteKReady, kSiteKEmpty, kSiteVFull, kSiteVEmpty,
  kSiteSFull, kSitePReady, kSiteQReady, kSiteOFinal, kSiteDrain, kSiteRelay
};

struct Ctl {
  uint64_t q_full[kQTiles];
  uint64_t q_ready[kQTiles];
  uint64_t k_full[kMaxStages];
  uint64_t k_ready[kMaxStages];
  uint64_t k_empty[kMaxStages];
  uint64_t v_full[kMaxStages];
  uint64_t v_empty[kMaxStages];
  uint64_t s_full[kQTiles];
  uint64_t p_ready[kQTiles];
  uint64_t o_final;
  uint32_t tmem_base;
  int abort_flag;
};

// Division of a non-negative 32-bit integer below 2^31 by an invariant divisor d >= 1:
// q = (umulhi(n, m) + n) >> s with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1
// (Granlund and Montgomery, "Division by invariant integers using multiplication", 1994).
struct FastDiv {
  uint32_t m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;
  const uint64_t m = ((1ull << 32) * ((1ull << s) - d)) / d + 1;
  return FastDiv{static_cast<uint32_t>(m), s};
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
  return (__umulhi(n, f.m) + n) >> f.s;
}

struct Params {
  int B, H, N, Hg, Wg, HgWg;
  // Optional block mask: bit kb of word kb/32 of row (b, h, query block) selects key tile kb.
  // Optional active-query subset: query rows are the tokens q_index[b * q_index_b_stride + i],
  // i < Nq, gathered from q and scattered back into out / lse.
  const int* q_index;          // nullptr: every token, in order
  int Nq;                      // query rows per (b, h)
  long long q_index_b_stride;  // entries between consecutive batches' lists (0: shared list)
  const __nv_bfloat16* q;      // q itself, for the gather
  int withhold_kv;             // testing only: the producer issues no K/V copy (waits expire)
  int q_prerot;                // Q arrives rotated and scaled (fp16, from the prepass) via TMA
  FastDiv div_H, div_N, div_HgWg, div_Wg;   // the prepass's row -> token -> (t, h, w) splits
  const uint32_t* kv_mask;     // nullptr: every key tile
  int mask_words;              // words per query block
  long long mask_bh_stride;    // words between consecutive (b, h) masks (0: one shared mask)
  int half_t, half_h, half_w;
  int off_h, off_w;            // table offsets of the h and w blocks (entries)
  int table_entries;
  int table_in_smem;
  int n_qblk;                  // CTAs per (b, h)
  int ctl_off;                 // byte offset of Ctl in the aligned dynamic smem
  float scale_log2;            // scale * log2(e)
  float omega[64];             // rotary frequency of each channel pair (pairs past d/2 unused)
  const float2* table;
  __nv_bfloat16* out;
  float* lse;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Row maximum of one 128-column score row: 16 independent 3-input max chains, then a short tree.
__device__ __forceinline__ float row_max128(const uint32_t (&s)[128]) {
  float mx16[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    mx16[i] = fmax3(__uint_as_float(s[i]), __uint_as_float(s[i + 16]), __uint_as_float(s[i + 32]));
#pragma unroll
  for (int i = 0; i < 16; ++i)
    mx16[i] = fmax3(mx16[i], __uint_as_float(s[i + 48]), __uint_as_float(s[i + 64]));
#pragma unroll
  for (int i = 0; i < 16; ++i)
    mx16[i] = fmax3(mx16[i], __uint_as_float(s[i + 80]), __uint_as_float(s[i + 96]));
#pragma unroll
  for (int i = 0; i < 16; ++i) mx16[i] = fmaxf(mx16[i], __uint_as_float(s[i + 112]));
#pragma unroll
  for (int i = 0; i < 5; ++i) mx16[i] = fmax3(mx16[i], mx16[i + 5], mx16[i + 10]);
  return fmax3(fmax3(mx16[0], mx16[1], mx16[2]), fmax3(mx16[3], mx16[4], mx16[15]), -INFINITY);
}

// p = 2^(s - m) for one 128-column row (scores in log2 units), packed to bf16 pairs in pk;
// returns the row sum of the fp32 p (four packed accumulators).
__device__ __forceinline__ float exp_row128(const uint32_t (&s)[128], float m, uint32_t (&pk)[64]) {
  const uint64_t negm2 = f32x2(-m, -m);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int e2 = 0; e2 < 64; ++e2) {
    const uint64_t a = fadd2(f32x2(__uint_as_float(s[2 * e2]), __uint_as_float(s[2 * e2 + 1])), negm2);
    float a0, a1;
    f32x2_split(a, a0, a1);
    const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
    acc[e2 & 3] = fadd2(acc[e2 & 3], f32x2(p0, p1));
    pk[e2] = pack_bf16x2(p0, p1);
  }
  float l0, l1;
  f32x2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), l0, l1);
  return l0 + l1;
}

// Round to fp16 with saturation to +-65504 (no infinities); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Bounded wait used on the way out: ignores the abort flag so that copies / MMAs that are
// still in flight finish before shared or tensor memory is released.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&g_error_word, 0u, 1u | (static_cast<unsigned>(kSiteDrain) << 8));
      return;
    }
  }
}

// S(tmem) = A(smem, 128 x 128, K-major) * B(smem, 128 x 128, K-major)^T in 8 steps of K=16.
// Each operand is two 16 KB halves (channels 0-63, 64-127); inside a 128-byte swizzled
// half, K step kk starts 32 bytes further on.
// Called by the whole MMA warp; one elected lane issues.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem,
                                         uint32_t idesc, bool accumulate = false) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss_warp(d_tmem, smem_desc_sw128(a_smem + off, 16, 1024),
                smem_desc_sw128(b_smem + off, 16, 1024), idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// O(tmem) (+)= P(tmem, 128 x 128 bf16) * V(smem, 128 keys x 128 channels, channel-contiguous).
// V is the MN-major B operand: 64-channel halves 16 KB apart (leading offset), 8-key groups
// 1 KB apart (stride offset); K step kk covers keys 16kk..16kk+15 = 2 KB further on.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    mma_ts_warp(d_tmem, p_tmem + kk * 8, smem_desc_sw128(v_smem + kk * 2048, kHalfBytes, 1024),
                idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Pair forms (rank-0 CTA of a pair only).  QK: A = this pair's Q tile (each CTA's 128 rows), B =
// a K tile whose keys 0-63 sit in rank 0's stage and 64-127 in rank 1's, each stage two 8 KB
// halves (channels 0-63, 64-127) of 64 rows x 128 bytes.  PV: A = P from each CTA's tensor
// memory, B = V with channels 0-63 in rank 0's stage and 64-127 in rank 1's (128 keys x 128
// bytes each, MN-major).  M = 256, N = 128 in both.
__device__ __forceinline__ void issue_qk_pair(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem,
                                              uint32_t idesc, bool accumulate = false) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t a_off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    const uint32_t b_off = (kk >> 2) * (kHalfBytes / 2) + (kk & 3) * 32;
    mma_ss_pair_warp(d_tmem, smem_desc_sw128(a_smem + a_off, 16, 1024),
                     smem_desc_sw128(b_smem + b_off, 16, 1024), idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}
__device__ __forceinline__ void issue_pv_pair(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                              uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    mma_ts_pair_warp(d_tmem, p_tmem + kk * 8, smem_desc_sw128(v_smem + kk * 2048, kHalfBytes, 1024),
                     idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Which rotary pairs a thread owns.  Thread t of the 128 RoPE threads always touches 16-byte
// chunk (t & 15) of a 256-byte row, i.e. pairs 4*(t&15) .. +3, so their axes and table
// columns are fixed per thread.
struct RopeLane {
  int tab_base[4];   // entry of position 0 for each of the thread's pairs
  int tab_stride[4]; // entries per position step on that pair's axis
  int axis[4];       // 0 = t, 1 = h, 2 = w
  float omega[4];    // rotary frequency of each pair
};

__device__ __forceinline__ RopeLane make_rope_lane(int c16, int half_t, int half_h, int half_w,
                                                   int off_h, int off_w, const float* omega) {
  RopeLane L;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int pr = c16 * 4 + e;
    L.omega[e] = omega[pr];
    if (pr < half_t) {
      L.axis[e] = 0; L.tab_base[e] = pr; L.tab_stride[e] = half_t;
    } else if (pr < half_t + half_h) {
      L.axis[e] = 1; L.tab_base[e] = off_h + (pr - half_t); L.tab_stride[e] = half_h;
    } else {
      L.axis[e] = 2; L.tab_base[e] = off_w + (pr - half_t - half_h); L.tab_stride[e] = half_w;
    }
  }
  return L;
}

// Rotate the 4 pairs of one 16-byte chunk (bf16 in) of a token at grid position (pt,ph,pw)
// and multiply by qs (scale*log2(e) for Q, 1 for K); returns the fp16 result and folds
// |result| into amax.
template <bool kLo, bool kSinCos = false>
__device__ __forceinline__ uint4 rotate_chunk(uint4 x, const RopeLane& L, int pt, int ph, int pw,
                                              const float2* __restrict__ tab, float& amax,
                                              uint4* lo_out = nullptr, float qs = 1.f) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t wl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int pos = L.axis[e] == 0 ? pt : (L.axis[e] == 1 ? ph : pw);
    float2 cs;
    if constexpr (kSinCos) {
      // angle and its cosine/sine on the special-function unit instead of a table lookup in
      // shared memory (absolute error ~1e-6 for the angles of a video grid, far below the
      // fp16 rounding of the result)
      __sincosf(static_cast<float>(pos) * L.omega[e], &cs.y, &cs.x);
    } else {
      cs = tab[L.tab_base[e] + pos * L.tab_stride[e]];
    }
    cs.x *= qs;
    cs.y *= qs;
    const float x0 = __uint_as_float(w[e] << 16);
    const float x1 = __uint_as_float(w[e] & 0xffff0000u);
    const float y0 = fmaf(x0, cs.x, -x1 * cs.y);
    const float y1 = fmaf(x0, cs.y, x1 * cs.x);
    amax = fmax3(amax, fabsf(y0), fabsf(y1));
    w[e] = pack_f16x2_sat(y0, y1);
    if (kLo) {
      const __half2 hi = *reinterpret_cast<const __half2*>(&w[e]);
      wl[e] = pack_f16x2_sat(y0 - __low2float(hi), y1 - __high2float(hi));
    }
  }
  if (kLo) *lo_out = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rotate one 128-row tile in place (bf16 in, fp16 out, swizzled halves).  Thread t handles
// chunk (t & 15) of rows (t >> 4) + 8*it; the 8 threads sharing a row hit 8 distinct
// 16-byte bank groups.
template <bool kLo, bool kSinCos = false, int kRows = kBM, int kHalfStride = kHalfBytes>
__device__ __forceinline__ float rope_tile(const Params& p, const RopeLane& L, int t, uint8_t* tile,
                                           int n_first, const float2* __restrict__ tab, float qs,
                                           uint8_t* lo_tile = nullptr) {
  float amax = 0.f;
  const int c16 = t & 15;
  const int rsub = t >> 4;
  const uint32_t chunk_off = (c16 >> 3) * kHalfStride + rsub * 128 + (((c16 & 7) ^ rsub) << 4);
  int n = n_first + rsub;
  if (n >= p.N) return amax;
  int pt = n / p.HgWg;
  int rem = n - pt * p.HgWg;
  int ph = rem / p.Wg;
  int pw = rem - ph * p.Wg;
#pragma unroll 2
  for (int it = 0; it < kRows / 8; ++it) {
    if (n >= p.N) break;
    // explicit 16-byte shared-memory accesses (the tile pointer is generic here): 4 % faster
    // than the generic accesses in the fused mode on CTA pairs
    const uint32_t a = smem_addr(tile + chunk_off + it * 1024);
    const uint4 y = rotate_chunk<kLo, kSinCos>(ld_shared_v4(a), L, pt, ph, pw, tab, amax,
                             kLo ? reinterpret_cast<uint4*>(lo_tile + chunk_off + it * 1024) : nullptr, qs);
    st_shared_v4(a, y);
    n += 8;
    pw += 8;
    while (pw >= p.Wg) { pw -= p.Wg; ++ph; }
    while (ph >= p.Hg) { ph -= p.Hg; ++pt; }
  }
  return amax;
}

// The key tiles a CTA visits, in increasing order: all nkv of them, or the tiles whose bit is
// set in its mask row (bits at or beyond nkv are ignored).  Every role walks the same sequence.
struct TileCursor {
  const uint32_t* row;   // nullptr: dense
  int nkv, word, words;
  uint32_t bits;
  int t;
  __device__ __forceinline__ uint32_t word_bits(int w) const {
    uint32_t x = __ldg(row + w);
    const int hi = nkv - 32 * w;            // valid bits in this word
    return hi >= 32 ? x : (x & ((1u << hi) - 1u));
  }
  __device__ __forceinline__ void init(const uint32_t* r, int n_kv, int n_words) {
    row = r; nkv = n_kv; words = n_words; word = 0; t = 0;
    bits = row ? word_bits(0) : 0u;
  }
  __device__ __forceinline__ int count() const {
    if (!row) return nkv;
    int c = 0;
    for (int w = 0; w < words; ++w) c += __popc(word_bits(w));
    return c;
  }
  // Next tile index; only called count() times.
  __device__ __forceinline__ int next() {
    if (!row) return t++;
    while (bits == 0) bits = word_bits(++word);
    const int b = __ffs(bits) - 1;
    bits &= bits - 1u;
    return word * 32 + b;
  }
};

// Gather 128 query rows (tokens q_index[row_base + row]) straight from q, rotate each at its
// own grid position and store them fp16 into a swizzled tile (rows past Nq, or with an index
// outside [0, N), become zeros; bad indices also raise error bit 4).  Same thread-to-chunk
// assignment as rope_tile.
template <bool kLo>
__device__ __forceinline__ float rope_gather_tile(const Params& p, const RopeLane& L, int t,
                                                  uint8_t* tile, const int* idx, int row_base,
                                                  int b, int h, const float2* __restrict__ tab, float qs,
                                                  uint8_t* lo_tile = nullptr) {
  float amax = 0.f;
  const int c16 = t & 15;
  const int rsub = t >> 4;
  const uint32_t chunk_off = (c16 >> 3) * kHalfBytes + rsub * 128 + (((c16 & 7) ^ rsub) << 4);
#pragma unroll 2
  for (int it = 0; it < kBM / 8; ++it) {
    const int i = row_base + it * 8 + rsub;
    int n = i < p.Nq ? __ldg(idx + i) : -1;
    if (i < p.Nq && (n < 0 || n >= p.N)) {
      atomicOr(&g_error_word, 4u);
      n = -1;
    }
    uint4 y = make_uint4(0u, 0u, 0u, 0u), ylo = y;
    if (n >= 0) {
      const int pt = n / p.HgWg;
      const int rem = n - pt * p.HgWg;
      const int ph = rem / p.Wg;
      const int pw = rem - ph * p.Wg;
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(
          p.q + ((static_cast<size_t>(b) * p.N + n) * p.H + h) * kD + c16 * 8));
      y = rotate_chunk<kLo>(x, L, pt, ph, pw, tab, amax, &ylo, qs);
    }
    *reinterpret_cast<uint4*>(tile + chunk_off + it * 1024) = y;
    if (kLo) *reinterpret_cast<uint4*>(lo_tile + chunk_off + it * 1024) = ylo;
  }
  return amax;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_klo,
               const __grid_constant__ CUtensorMap tm_qlo, const __grid_constant__ CUtensorMap tm_out,
               const Params p) {
  using Lo = Layout<kMode>;
  constexpr bool kFusedK = Lo::kFusedK;
  constexpr bool kSplit = Lo::kSplit;
  constexpr bool kPair = Lo::kPair;
  constexpr int kKStages = Lo::kKStages;
  constexpr int kVStages = Lo::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + p.ctl_off);
  float2* tab_s = reinterpret_cast<float2*>(smem + Lo::kOffTab);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int qblk = blockIdx.x % p.n_qblk;
  const int bh = blockIdx.x / p.n_qblk;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int q0 = qblk * kRowsPerCta;               // first query row of this CTA
  const int* q_idx = p.q_index ? p.q_index + static_cast<long long>(b) * p.q_index_b_stride : nullptr;
  const int nkv_all = (p.N + kBN - 1) / kBN;
  const uint32_t* mask_row =
      p.kv_mask ? p.kv_mask + (static_cast<long long>(bh) * p.mask_bh_stride +
                               static_cast<long long>(qblk) * p.mask_words)
                : nullptr;
  TileCursor cur;
  cur.init(mask_row, nkv_all, p.mask_words);
  const int nkv = cur.count();              // key tiles this CTA visits (steps j = 0..nkv-1)

  const uint32_t sQ = smem_addr(smem + Lo::kOffQ);
  const uint32_t sK = smem_addr(smem + Lo::kOffK);
  const uint32_t sV = smem_addr(smem + Lo::kOffV);
  // CTA pair: rank 0 (the leader) issues every MMA; its q/k/v "full" barriers also count one
  // relayed arrival from rank 1 once rank 1's own half has landed, and its P-ready barriers
  // one arrival from each of rank 1's softmax warps.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0u;
  // With the fused K rotation the leader waits for the rotated tiles instead (its q/k "ready"
  // barriers count one arrival from each of rank 1's RoPE warps), so rank 1 relays V only.
  const uint32_t full_count = (kPair && leader) ? 2u : 1u;
  const uint32_t qk_full_count = kFusedK ? 1u : full_count;
  const uint32_t ready_count = kPair ? 128 + 4 : 128;

  if (tid == 0) {
    for (int i = 0; i < kQTiles; ++i) {
      mbar_init(smem_addr(&ctl->q_full[i]), qk_full_count);
      mbar_init(smem_addr(&ctl->q_ready[i]), ready_count);
      mbar_init(smem_addr(&ctl->s_full[i]), 1);
      mbar_init(smem_addr(&ctl->p_ready[i]), kPair ? 128 + 4 : 128);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_addr(&ctl->k_full[s]), qk_full_count);
      mbar_init(smem_addr(&ctl->k_ready[s]), ready_count);
      mbar_init(smem_addr(&ctl->k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_addr(&ctl->v_full[s]), full_count);
      mbar_init(smem_addr(&ctl->v_empty[s]), 1);
    }
    mbar_init(smem_addr(&ctl->o_final), 1);
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_addr(&ctl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  if (kFusedK && p.table_in_smem) {
    for (int i = tid; i < p.table_entries; i += kThreads) tab_s[i] = p.table[i];
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();   // both CTAs' barriers exist before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp >= 12) {
    regs_decrease<Lo::kRegsCtl>();
    if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (kSplit) tma_prefetch_desc(&tm_klo);
      const bool q_lo = kSplit && p.q_prerot;               // Q remainders come from the prepass too
      if (q_lo) tma_prefetch_desc(&tm_qlo);
      for (int i = 0; i < kQTiles && q_idx == nullptr; ++i) {   // a query subset is gathered by WG2
        const uint32_t bar = smem_addr(&ctl->q_full[i]);
        mbar_arrive_expect_tx(bar, q_lo ? 2 * kTileBytes : kTileBytes);
        const uint32_t dst = sQ + i * kTileBytes;
        tma_load_4d(dst, &tm_q, bar, 0, h, q0 + i * kBM, b);
        tma_load_4d(dst + kHalfBytes, &tm_q, bar, 64, h, q0 + i * kBM, b);
        if (q_lo) {
          const uint32_t dlo = smem_addr(smem + Lo::kOffQlo) + i * kTileBytes;
          tma_load_4d(dlo, &tm_qlo, bar, 0, h, q0 + i * kBM, b);
          tma_load_4d(dlo + kHalfBytes, &tm_qlo, bar, 64, h, q0 + i * kBM, b);
        }
      }
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nkv && !p.withhold_kv; ++j) {
        const int kt = cur.next();          // key tile of step j
        const int ks = j % kKStages, ku = j / kKStages;
        if (ku > 0 && !mbar_wait(smem_addr(&ctl->k_empty[ks]), (ku - 1) & 1, abort_flag, kSiteKEmpty))
          break;
        if constexpr (kPair) {
          // this CTA's 64 keys of the tile (the K maps have 64-token boxes here): hi, then lo
          const uint32_t bar = smem_addr(&ctl->k_full[ks]);
          mbar_arrive_expect_tx(bar, Lo::kKStageBytes);
          const uint32_t dst = sK + ks * Lo::kKStageBytes;
          const int row = kt * kBN + static_cast<int>(rank) * (kBN / 2);
          tma_load_4d(dst, &tm_k, bar, 0, h, row, b);
          tma_load_4d(dst + kHalfBytes / 2, &tm_k, bar, 64, h, row, b);
          if (kSplit) {
            tma_load_4d(dst + kTileBytes / 2, &tm_klo, bar, 0, h, row, b);
            tma_load_4d(dst + kTileBytes / 2 + kHalfBytes / 2, &tm_klo, bar, 64, h, row, b);
          }
          k_issued = j + 1;
        } else {
          const uint32_t bar = smem_addr(&ctl->k_full[ks]);
          mbar_arrive_expect_tx(bar, Lo::kKStageBytes);
          const uint32_t dst = sK + ks * Lo::kKStageBytes;
          tma_load_4d(dst, &tm_k, bar, 0, h, kt * kBN, b);
          tma_load_4d(dst + kHalfBytes, &tm_k, bar, 64, h, kt * kBN, b);
          if (kSplit) {
            tma_load_4d(dst + kTileBytes, &tm_klo, bar, 0, h, kt * kBN, b);
            tma_load_4d(dst + kTileBytes + kHalfBytes, &tm_klo, bar, 64, h, kt * kBN, b);
          }
          k_issued = j + 1;
        }
        const int vs = j % kVStages, vu = j / kVStages;
        if (vu > 0 && !mbar_wait(smem_addr(&ctl->v_empty[vs]), (vu - 1) & 1, abort_flag, kSiteVEmpty))
          break;
        {
          const uint32_t bar = smem_addr(&ctl->v_full[vs]);
          mbar_arrive_expect_tx(bar, Lo::kVStageBytes);
          const uint32_t dst = sV + vs * Lo::kVStageBytes;
          if constexpr (kPair) {
            tma_load_4d(dst, &tm_v, bar, static_cast<int>(rank) * 64, h, kt * kBN, b);   // this CTA's 64 channels
          } else {
            tma_load_4d(dst, &tm_v, bar, 0, h, kt * kBN, b);
            tma_load_4d(dst + kHalfBytes, &tm_v, bar, 64, h, kt * kBN, b);
          }
          v_issued = j + 1;
        }
      }
      // Let every copy this thread started land before the CTA can retire.
      for (int i = 0; i < kQTiles && q_idx == nullptr; ++i) drain_wait(smem_addr(&ctl->q_full[i]), 0);
      for (int s = 0; s < kKStages; ++s) {
        const int uses = k_issued > s ? (k_issued - 1 - s) / kKStages + 1 : 0;
        if (uses > 0) drain_wait(smem_addr(&ctl->k_full[s]), (uses - 1) & 1);
      }
      for (int s = 0; s < kVStages; ++s) {
        const int uses = v_issued > s ? (v_issued - 1 - s) / kVStages + 1 : 0;
        if (uses > 0) drain_wait(smem_addr(&ctl->v_full[s]), (uses - 1) & 1);
      }
    } else if (kPair && warp == 13 && leader) {
      // ---------------------------------------------------------- MMA issuer of a CTA pair:
      // the same issue order as below with cta_group::2 MMAs over both CTAs' rows and halves;
      // every barrier it waits on also counts arrivals from rank 1.
      constexpr uint32_t kIdQK = idesc_f16kind_f32acc(2 * kBM, kBN, 0, 0);
      constexpr uint32_t kIdPV = idesc_f16kind_f32acc(2 * kBM, kD, 1, 1);
      const uint32_t tS0 = tmem + 0, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      const uint64_t* qbar = kFusedK ? ctl->q_ready : ctl->q_full;
      bool ok = mbar_wait(smem_addr(&qbar[0]), 0, abort_flag, kSiteQReady) &&
                mbar_wait(smem_addr(&qbar[1]), 0, abort_flag, kSiteQReady);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after_sync();
      auto k_wait = [&](int jj) {
        const int kss = jj % kKStages;
        const uint32_t kbar = kFusedK ? smem_addr(&ctl->k_ready[kss]) : smem_addr(&ctl->k_full[kss]);
        return mbar_wait(kbar, (jj / kKStages) & 1, abort_flag, kFusedK ? kSiteKReady : kSiteKFull);
      };
      if (ok && nkv > 0) ok = __all_sync(0xffffffffu, k_wait(0));
      for (int j = 0; ok && j < nkv; ++j) {
        const int ks = j % kKStages;
        tc_fence_after_sync();
        const uint32_t kst = sK + ks * Lo::kKStageBytes;
        const uint32_t sQlo = smem_addr(smem + Lo::kOffQlo);
        issue_qk_pair(tS0, sQ, kst, kIdQK);
        if (kSplit) {
          issue_qk_pair(tS0, sQ, kst + kTileBytes / 2, kIdQK, true);     // Qhi Klo
          issue_qk_pair(tS0, sQlo, kst, kIdQK, true);                    // Qlo Khi
        }
        mma_commit_pair_warp(smem_addr(&ctl->s_full[0]));
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->p_ready[1]), (j - 1) & 1, abort_flag,
                                                         kSitePReady));
          if (!ok) break;
          tc_fence_after_sync();
          const int pvs = (j - 1) % kVStages;
          issue_pv_pair(tO1, tS1, sV + pvs * Lo::kVStageBytes, kIdPV, j - 1 > 0);
          mma_commit_pair_warp(smem_addr(&ctl->v_empty[pvs]));
        }
        issue_qk_pair(tS1, sQ + kTileBytes, kst, kIdQK);
        if (kSplit) {
          issue_qk_pair(tS1, sQ + kTileBytes, kst + kTileBytes / 2, kIdQK, true);
          issue_qk_pair(tS1, sQlo + kTileBytes, kst, kIdQK, true);
        }
        mma_commit_pair_warp(smem_addr(&ctl->s_full[1]));
        mma_commit_pair_warp(smem_addr(&ctl->k_empty[ks]));
        const int vs = j % kVStages;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(smem_addr(&ctl->v_full[vs]), (j / kVStages) & 1, abort_flag, kSiteVFull) &&
                        (j + 1 >= nkv || k_wait(j + 1)) &&
                        mbar_wait(smem_addr(&ctl->p_ready[0]), j & 1, abort_flag, kSitePReady));
        if (!ok) break;
        tc_fence_after_sync();
        issue_pv_pair(tO0, tS0, sV + vs * Lo::kVStageBytes, kIdPV, j > 0);
      }
      if (ok && nkv > 0) {
        const int jl = nkv - 1;
        if (__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->p_ready[1]), jl & 1, abort_flag, kSitePReady))) {
          tc_fence_after_sync();
          issue_pv_pair(tO1, tS1, sV + (jl % kVStages) * Lo::kVStageBytes, kIdPV, jl > 0);
        }
      }
      mma_commit_pair_warp(smem_addr(&ctl->o_final));
      drain_wait(smem_addr(&ctl->o_final), 0);
    } else if (kPair && warp == 13 && !leader) {
      // rank 1: the leader's final commit also arrives here; see it land before this CTA can
      // retire (the softmax warps skip their wait for it after an abort)
      drain_wait(smem_addr(&ctl->o_final), 0);
    } else if (kPair && warp == 14 && lane == 0 && !leader) {
      // ---------------------------------------------------------- relay (rank 1 of a pair):
      // tells the leader, through one remote arrival per phase, that this CTA's Q tiles and
      // its half of each K/V stage have landed.
      bool ok = true;
      for (int i = 0; ok && i < kQTiles && !kFusedK; ++i) {
        ok = mbar_wait(smem_addr(&ctl->q_full[i]), 0, abort_flag, kSiteRelay);
        if (ok) mbar_arrive_remote(mapa_shared(smem_addr(&ctl->q_full[i]), 0));
      }
      for (int j = 0; ok && j < nkv && !p.withhold_kv; ++j) {
        const int ks = j % kKStages, vs = j % kVStages;
        if constexpr (!kFusedK) {
          if (!(ok = mbar_wait(smem_addr(&ctl->k_full[ks]), (j / kKStages) & 1, abort_flag, kSiteRelay))) break;
          mbar_arrive_remote(mapa_shared(smem_addr(&ctl->k_full[ks]), 0));
        }
        if (!(ok = mbar_wait(smem_addr(&ctl->v_full[vs]), (j / kVStages) & 1, abort_flag, kSiteRelay))) break;
        mbar_arrive_remote(mapa_shared(smem_addr(&ctl->v_full[vs]), 0));
      }
    } else if (!kPair && warp == 13) {
      // ---------------------------------------------------------- MMA issuer (whole warp runs
      // the loop so descriptor arithmetic stays warp-uniform; one elected lane issues)
      constexpr uint32_t kIdQK = idesc_f16kind_f32acc(kBM, kBN, 0, 0);   // fp16 Q', K'
      constexpr uint32_t kIdPV = idesc_f16kind_f32acc(kBM, kD, 1, 1);   // bf16 P, V (MN-major)
      const uint32_t tS0 = tmem + 0, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
      // Q tiles are ready when their copies land (pre-rotated by the prepass) or once WG2 has
      // rotated them in shared memory.
      const uint64_t* qbar = p.q_prerot ? ctl->q_full : ctl->q_ready;
      bool ok = mbar_wait(smem_addr(&qbar[0]), 0, abort_flag, kSiteQReady) &&
                mbar_wait(smem_addr(&qbar[1]), 0, abort_flag, kSiteQReady);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after_sync();
      // K tile j is ready: waited for at the top of step j with a one-stage ring (split mode:
      // K(j+1) lands only after S1(j) frees the stage), else before PV0(j-1) so that S0(j)
      // follows PV0(j-1) without a barrier wait in between.
      auto k_wait = [&](int jj) {
        const int kss = jj % kKStages;
        const uint32_t kbar = kFusedK ? smem_addr(&ctl->k_ready[kss]) : smem_addr(&ctl->k_full[kss]);
        return mbar_wait(kbar, (jj / kKStages) & 1, abort_flag, kFusedK ? kSiteKReady : kSiteKFull);
      };
      if (!kSplit && ok && nkv > 0) ok = __all_sync(0xffffffffu, k_wait(0));
      for (int j = 0; ok && j < nkv; ++j) {
        const int ks = j % kKStages;
        if (kSplit) {
          ok = __all_sync(0xffffffffu, k_wait(j));
          if (!ok) break;
        }
        tc_fence_after_sync();
        const uint32_t kt = sK + ks * Lo::kKStageBytes;
        const uint32_t sQlo = smem_addr(smem + Lo::kOffQlo);
        issue_qk(tS0, sQ, kt, kIdQK);
        if (kSplit) {
          issue_qk(tS0, sQ, kt + kTileBytes, kIdQK, true);     // Qhi Klo
          issue_qk(tS0, sQlo, kt, kIdQK, true);                // Qlo Khi
        }
        mma_commit_warp(smem_addr(&ctl->s_full[0]));
        if (j > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->p_ready[1]), (j - 1) & 1, abort_flag,
                                                 kSitePReady));
          if (!ok) break;
          tc_fence_after_sync();
          const int pvs = (j - 1) % kVStages;
          issue_pv(tO1, tS1, sV + pvs * kTileBytes, kIdPV, j - 1 > 0);
          mma_commit_warp(smem_addr(&ctl->v_empty[pvs]));
        }
        issue_qk(tS1, sQ + kTileBytes, kt, kIdQK);
        if (kSplit) {
          issue_qk(tS1, sQ + kTileBytes, kt + kTileBytes, kIdQK, true);
          issue_qk(tS1, sQlo + kTileBytes, kt, kIdQK, true);
        }
        mma_commit_warp(smem_addr(&ctl->s_full[1]));
        mma_commit_warp(smem_addr(&ctl->k_empty[ks]));
        const int vs = j % kVStages;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(smem_addr(&ctl->v_full[vs]), (j / kVStages) & 1, abort_flag, kSiteVFull) &&
                        (kSplit || j + 1 >= nkv || k_wait(j + 1)) &&
                        mbar_wait(smem_addr(&ctl->p_ready[0]), j & 1, abort_flag, kSitePReady));
        if (!ok) break;
        tc_fence_after_sync();
        issue_pv(tO0, tS0, sV + vs * kTileBytes, kIdPV, j > 0);
      }
      if (ok && nkv > 0) {
        const int jl = nkv - 1;
        if (__all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->p_ready[1]), jl & 1, abort_flag, kSitePReady))) {
          tc_fence_after_sync();
          issue_pv(tO1, tS1, sV + (jl % kVStages) * kTileBytes, kIdPV, jl > 0);
        }
      }
      mma_commit_warp(smem_addr(&ctl->o_final));
      drain_wait(smem_addr(&ctl->o_final), 0);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ RoPE on Q (and K tiles)
    regs_decrease<Lo::kRegsRope>();
    const int t = tid - 256;
    const float2* tab = (kFusedK && p.table_in_smem) ? tab_s : p.table;
    const RopeLane L = make_rope_lane(t & 15, p.half_t, p.half_h, p.half_w, p.off_h, p.off_w, p.omega);
    bool ok = true;
    float amax = 0.f;
    // This thread's rotated chunks are in place: make them visible to the tensor cores and
    // arrive (rank 1 of a pair: one arrival per warp on the leader's barrier).
    auto rotated = [&](uint64_t* bar) {
      fence_proxy_async_smem();
      if (!kPair || leader) {
        mbar_arrive(smem_addr(bar));
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_release(mapa_shared(smem_addr(bar), 0));
      }
    };
    for (int i = 0; i < kQTiles && ok && !p.q_prerot; ++i) {
      if (q_idx) {
        amax = fmaxf(amax, rope_gather_tile<kSplit>(p, L, t, smem + Lo::kOffQ + i * kTileBytes, q_idx,
                                                    q0 + i * kBM, b, h, tab, p.scale_log2,
                                                    smem + Lo::kOffQlo + i * kTileBytes));
      } else {
        // warp-uniform, so that a warp of rank 1 reaches its per-warp arrival together
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->q_full[i]), 0, abort_flag, kSiteQFull))))
          break;
        // CTA pairs with the fused K rotation take on-the-fly cosines/sines (their shared memory
        // holds no table)
        amax = fmaxf(amax, rope_tile<kSplit, kPair && kFusedK>(p, L, t, smem + Lo::kOffQ + i * kTileBytes, q0 + i * kBM,
                                                    tab, p.scale_log2, smem + Lo::kOffQlo + i * kTileBytes));
      }
      rotated(&ctl->q_ready[i]);
    }
    if (kFusedK) {
      for (int j = 0; ok && j < nkv; ++j) {
        const int kt = cur.next();
        const int ks = j % kKStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->k_full[ks]), (j / kKStages) & 1,
                                                      abort_flag, kSiteKFull))))
          break;
        uint8_t* kst = smem + Lo::kOffK + ks * Lo::kKStageBytes;
        if constexpr (kPair)   // this CTA's 64 keys of the tile, 64-channel halves 8 KB apart
          amax = fmaxf(amax, rope_tile<false, true, kBN / 2, kHalfBytes / 2>(
                                 p, L, t, kst, kt * kBN + static_cast<int>(rank) * (kBN / 2), tab, 1.f));
        else
          amax = fmaxf(amax, rope_tile<false, true>(p, L, t, kst, kt * kBN, tab, 1.f));
        rotated(&ctl->k_ready[ks]);
      }
    }
    if (!(amax <= 65504.f)) atomicOr(&g_error_word, 2u);
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    regs_increase<Lo::kRegsSoftmax>();
    const int qi = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_bits + 128 * qi;
    const uint32_t tO = tmem + lane_bits + 256 + 128 * qi;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int kt = cur.next();
      if (!(ok = mbar_wait(smem_addr(&ctl->s_full[qi]), j & 1, abort_flag, kSiteSFull))) break;
      tc_fence_after_sync();
      uint32_t s[128];
      tmem_ld128(tS, s);
      const int valid = p.N - kt * kBN;
      if (valid < kBN) {             // ragged last tile: keys beyond N weigh nothing
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (e >= valid) s[e] = 0xff800000u;
      }
      // Exponentials against the running maximum, kept when the row sum shows every p <= 256
      // (P then stays within the range the accumulators are sized for).  Otherwise (the first
      // tile, or a row whose scores rose) take the exact tile maximum, move the running
      // maximum there, rescale l (and O below) and redo the row; S is still intact in TMEM
      // because P has not been stored yet.
      uint32_t pk[64];
      float l_tile = exp_row128(s, m_run, pk);
      bool resc = false;
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, !(l_tile <= 256.f))) {
        tmem_ld128(tS, s);
        if (valid < kBN) {
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e >= valid) s[e] = 0xff800000u;
        }
        const float m_new = fmaxf(m_run, row_max128(s));
        resc = m_new > m_run;
        if (resc) {
          alpha = ex2_approx(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
        }
        l_tile = exp_row128(s, m_run, pk);
      }
      {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
        tmem_st32(tS, lo);
        tmem_st32(tS + 32, hi);
      }
      l_run += l_tile;
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        uint32_t r[32];
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          tmem_ld32(tO + ch * 32, r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tO + ch * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      if (!kPair || leader) {
        mbar_arrive(smem_addr(&ctl->p_ready[qi]));
      } else {
        // rank 1 of a pair: one arrival per warp on the leader's barrier, once all its lanes
        // have stored their rows of P
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_addr(&ctl->p_ready[qi]), 0));
      }
    }
    if (ok) ok = mbar_wait(smem_addr(&ctl->o_final), 0, abort_flag, kSiteOFinal);
    if (ok) {
      tc_fence_after_sync();
      const int i_row = q0 + qi * kBM + row;            // query row
      int n = i_row;                                    // its token
      bool live = i_row < p.Nq;
      if (q_idx) {
        n = live ? __ldg(q_idx + i_row) : 0;
        live = live && n >= 0 && n < p.N;
      }
      // A query block whose mask selects no key tile has no keys: out = 0, lse = -inf.
      const bool empty = nkv == 0;
      const float inv_l = empty ? 0.f : 1.f / l_run;
      __nv_bfloat16* orow = p.out + ((static_cast<size_t>(b) * p.N + (live ? n : 0)) * p.H + h) * kD;
      // Without a query subset the tile is staged in its Q buffer (free: every MMA that read
      // it has completed) in the 128-byte-swizzled layout and leaves through TMA below.
      uint8_t* stile = smem + Lo::kOffQ + qi * kTileBytes;
      uint32_t r[32];
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        if (empty) {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        } else {
          tmem_ld32(tO + ch * 32, r);
        }
        uint32_t pk[16];
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2)
          pk[e2] = pack_bf16x2(__uint_as_float(r[2 * e2]) * inv_l, __uint_as_float(r[2 * e2 + 1]) * inv_l);
        if (q_idx == nullptr) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = ch * 4 + u;            // 16-byte chunk of the row (8 channels)
            *reinterpret_cast<uint4*>(stile + (c >> 3) * kHalfBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        } else if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (q_idx == nullptr) fence_proxy_async_smem();
      if (live && p.lse != nullptr)
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.N + n] =
            empty ? -INFINITY : (m_run + __log2f(l_run)) * 0.69314718055994530942f;
    }
    if (q_idx == nullptr) {
      // Every thread of the warpgroup gets here (also after an abort), so the barrier cannot
      // strand anyone; one thread then stores the tile (rows past N are clipped by TMA).
      __syncwarp();
      named_barrier_sync(1 + qi, 128);
      const int r0 = q0 + qi * kBM;
      if (ok && (warp & 3) == 0 && lane == 0 && r0 < p.N) {
        const uint32_t src = smem_addr(smem + Lo::kOffQ + qi * kTileBytes);
        tma_store_4d(&tm_out, src, 0, h, r0, b);
        tma_store_4d(&tm_out, src + kHalfBytes, 64, h, r0, b);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();   // neither CTA leaves while the pair's MMAs may use it
  if (warp == 13) {
    tc_fence_after_sync();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

// Q/K prepass: rotate every token of K (blockIdx.y = 0) and of Q (blockIdx.y = 1, multiplied
// by scale*log2(e)) once: bf16 in, fp16 out, same [B, N, H, d] layout; with kLo the fp16
// remainders follow each tensor as a second [B, N, H, d] tensor.
// One thread per 16-byte chunk; the grid stride is a multiple of 16 chunks, so each thread
// keeps one chunk column (and its four rotary pairs) throughout.
template <bool kLo, bool kQ>
__device__ __forceinline__ void rope3d_prepass_body(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                    const Params& p, uint32_t n_chunks) {
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  const RopeLane L = make_rope_lane(static_cast<int>(c & 15), p.half_t, p.half_h, p.half_w,
                                    p.off_h, p.off_w, p.omega);
  const float qs = kQ ? p.scale_log2 : 1.f;
  float amax = 0.f;
  for (; c < n_chunks; c += stride) {
    const uint32_t row = c >> 4;                       // (b*N + n)*H + h
    const uint32_t bn = fast_div(row, p.div_H);         // b*N + n
    const uint32_t n = bn - fast_div(bn, p.div_N) * static_cast<uint32_t>(p.N);
    const int pt = static_cast<int>(fast_div(n, p.div_HgWg));
    const int rem = static_cast<int>(n) - pt * p.HgWg;
    const int ph = static_cast<int>(fast_div(static_cast<uint32_t>(rem), p.div_Wg));
    const int pw = rem - ph * p.Wg;
    const uint4 x = __ldg(src + c);
    dst[c] = rotate_chunk<kLo>(x, L, pt, ph, pw, p.table, amax, kLo ? dst + n_chunks + c : nullptr, qs);
  }
  if (!(amax <= 65504.f)) atomicOr(&g_error_word, 2u);
}

template <bool kLo>
__global__ void __launch_bounds__(256)
rope3d_qk_prepass(const uint4* __restrict__ k, uint4* __restrict__ kr, const uint4* __restrict__ q,
                  uint4* __restrict__ qr, const Params p, uint32_t n_chunks) {
  if (blockIdx.y == 0)
    rope3d_prepass_body<kLo, false>(k, kr, p, n_chunks);
  else
    rope3d_prepass_body<kLo, true>(q, qr, p, n_chunks);
}

void fill_params(const Problem& pr, Params* p) {
  *p = Params{};
  p->B = pr.B; p->H = pr.H; p->N = pr.N; p->Hg = pr.Hg; p->Wg = pr.Wg; p->HgWg = pr.Hg * pr.Wg;
  p->half_t = pr.half_t; p->half_h = pr.half_h; p->half_w = pr.half_w;
  p->off_h = pr.T * pr.half_t;
  p->off_w = p->off_h + pr.Hg * pr.half_h;
  p->table_entries = pr.table_entries;
  {
    const int halves[3] = {pr.half_t, pr.half_h, pr.half_w};
    int pair = 0;
    for (int a = 0; a < 3; ++a)
      for (int j = 0; j < halves[a] && pair < 64; ++j)
        p->omega[pair++] = static_cast<float>(std::pow(pr.theta, -2.0 * j / (2 * halves[a])));
  }
  p->scale_log2 = pr.scale * 1.4426950408889634f;
  p->table = pr.table;
  p->out = static_cast<__nv_bfloat16*>(pr.out);
  p->lse = pr.lse;
  p->q_index = pr.q_index;
  p->Nq = pr.q_index ? pr.Nq : pr.N;
  p->q_index_b_stride = pr.q_index_b_stride;
  p->q = static_cast<const __nv_bfloat16*>(pr.q);
  p->n_qblk = (p->Nq + kRowsPerCta - 1) / kRowsPerCta;
  p->withhold_kv = pr.withhold_kv;
  p->kv_mask = pr.kv_mask;
  p->mask_words = pr.mask_words;
  p->mask_bh_stride = pr.mask_bh_stride;
  p->div_H = make_fastdiv(static_cast<uint32_t>(pr.H));
  p->div_N = make_fastdiv(static_cast<uint32_t>(pr.N));
  p->div_HgWg = make_fastdiv(static_cast<uint32_t>(pr.Hg * pr.Wg));
  p->div_Wg = make_fastdiv(static_cast<uint32_t>(pr.Wg));
}

CUresult encode_bhnd(EncodeTiledFn encode, CUtensorMap* map, const void* base,
                     CUtensorMapDataType dtype, const Problem& pr, int box_tokens = kBN) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(pr.H),
                              static_cast<cuuint64_t>(pr.N), static_cast<cuuint64_t>(pr.B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * 2,
                                 static_cast<cuuint64_t>(pr.H) * kD * 2,
                                 static_cast<cuuint64_t>(pr.N) * pr.H * kD * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_tokens), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(map, dtype, 4, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int kMode>
cudaError_t launch_attn(const Problem& pr, Params p, const CUtensorMap* maps, cudaStream_t stream,
                        const char** what) {
  using Lo = Layout<kMode>;
  constexpr bool kFusedK = Lo::kFusedK;
  const int tab_bytes = ((pr.table_entries * 8) + 15) & ~15;
  const int ctl_bytes = (static_cast<int>(sizeof(Ctl)) + 15) & ~15;
  int smem = Lo::kOffTab + tab_bytes + ctl_bytes + 1024;
  if (kFusedK && !Lo::kPair && smem <= kMaxDynSmem) {
    p.table_in_smem = 1;
    p.ctl_off = Lo::kOffTab + tab_bytes;
  } else {
    p.table_in_smem = 0;
    p.ctl_off = Lo::kOffTab;
    smem = Lo::kOffTab + ctl_bytes + 1024;
  }
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_sm103<kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    *what = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  const long long grid = static_cast<long long>(pr.B) * pr.H * p.n_qblk;
  if (grid > 0x7fffffffLL) {
    *what = "grid too large";
    return cudaErrorInvalidValue;
  }
  if constexpr (Lo::kPair) {
    // clusters of two CTAs (consecutive query blocks of one (b, h); n_qblk is even)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_fwd_sm103<kMode>, maps[0], maps[1], maps[2], maps[3], maps[4],
                           maps[5], p);
    if (e != cudaSuccess) {
      *what = "attention kernel launch (CTA pairs) failed";
      return e;
    }
  } else {
    attn_fwd_sm103<kMode><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(maps[0], maps[1], maps[2],
                                                                                maps[3], maps[4], maps[5], p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) *what = "attention kernel launch failed";
  return e;
}

}  // namespace

cudaError_t read_and_clear_error_word_sm103(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned int));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
}

size_t prepass_workspace_bytes(const Problem& pr, bool split, bool with_q) {
  return static_cast<size_t>(pr.B) * pr.N * pr.H * kD * 2 * (split ? 2 : 1) * (with_q ? 2 : 1);
}

cudaError_t launch_attn_bf16_sm103(const Problem& pr, EncodeTiledFn encode, KMode mode,
                                   void* workspace, bool rotate_q_in_prepass, cudaStream_t stream,
                                   const char** what) {
  *what = nullptr;
  Params p;
  fill_params(pr, &p);
  CUtensorMap maps[6];
  const bool fused = mode == KMode::kFused || mode == KMode::kPairFused;
  const bool split = mode == KMode::kSplit || mode == KMode::kPairSplit;
  const bool pair = mode == KMode::kPair || mode == KMode::kPairSplit || mode == KMode::kPairFused;
  if (pair) {
    if (pr.q_index != nullptr || pr.kv_mask != nullptr) {
      *what = "CTA pairs take dense calls only";
      return cudaErrorInvalidValue;
    }
    p.n_qblk += p.n_qblk & 1;      // a pair's two CTAs share one (b, h)
  }
  const bool q_pre = !fused && rotate_q_in_prepass && pr.q_index == nullptr;
  p.q_prerot = q_pre ? 1 : 0;
  const void* kbase = pr.k;
  const void* klo = pr.k;
  const void* qbase = pr.q;
  const void* qlo = pr.q;
  if (!fused) {
    const size_t tb = prepass_workspace_bytes(pr, false, false);      // one fp16 tensor
    const size_t chunks = tb / 16;
    if (chunks >= 0x40000000ull) {
      *what = "Q/K prepass: tensor too large";
      return cudaErrorInvalidValue;
    }
    int sms = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (static_cast<long long>(chunks) + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(std::min<long long>(want, static_cast<long long>(sms) * 8));
    // Workspace: K' [K' lo] then, when Q is rotated here too, Q' [Q' lo].
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t* qws = ws + tb * (split ? 2 : 1);
    const dim3 grid(blocks, q_pre ? 2 : 1);
    if (split)
      rope3d_qk_prepass<true><<<grid, 256, 0, stream>>>(
          static_cast<const uint4*>(pr.k), reinterpret_cast<uint4*>(ws), static_cast<const uint4*>(pr.q),
          reinterpret_cast<uint4*>(qws), p, static_cast<uint32_t>(chunks));
    else
      rope3d_qk_prepass<false><<<grid, 256, 0, stream>>>(
          static_cast<const uint4*>(pr.k), reinterpret_cast<uint4*>(ws), static_cast<const uint4*>(pr.q),
          reinterpret_cast<uint4*>(qws), p, static_cast<uint32_t>(chunks));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      *what = "Q/K prepass launch failed";
      return e;
    }
    kbase = ws;
    klo = ws + tb;
    if (q_pre) {
      qbase = qws;
      qlo = qws + tb;
    }
  }
  const CUtensorMapDataType kdt = fused ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType qdt = q_pre ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (encode_bhnd(encode, &maps[0], qbase, qdt, pr) != CUDA_SUCCESS ||
      encode_bhnd(encode, &maps[1], kbase, kdt, pr, pair ? kBN / 2 : kBN) != CUDA_SUCCESS ||
      encode_bhnd(encode, &maps[2], pr.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pr) != CUDA_SUCCESS ||
      encode_bhnd(encode, &maps[3], split ? klo : kbase, kdt, pr, pair ? kBN / 2 : kBN) != CUDA_SUCCESS ||
      encode_bhnd(encode, &maps[4], split && q_pre ? qlo : qbase, qdt, pr) != CUDA_SUCCESS ||
      encode_bhnd(encode, &maps[5], pr.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pr) != CUDA_SUCCESS) {
    *what = "cuTensorMapEncodeTiled failed";
    return cudaErrorInvalidValue;
  }
  if (fused && pair) return launch_attn<kModePairFused>(pr, p, maps, stream, what);
  if (fused) return launch_attn<kModeFused>(pr, p, maps, stream, what);
  if (pair && split) return launch_attn<kModePairSplit>(pr, p, maps, stream, what);
  if (pair) return launch_attn<kModePair>(pr, p, maps, stream, what);
  if (split) return launch_attn<kModeSplit>(pr, p, maps, stream, what);
  return launch_attn<kModePrepass>(pr, p, maps, stream, what);
}

}  // namespace vdx
