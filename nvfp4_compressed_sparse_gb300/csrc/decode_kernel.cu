// sparse_mla_decode kernels: NVFP4 sparse MLA decode on sm_103a (tcgen05 + TMEM + TMA).
//
// What is computed ("Prime Inference", translated page, "Native NVFP4 sparse MLA
// decode kernel"; "Serving GLM-5.3 ...", "A kernel that reads four bits
// directly"): each query token reads only the cache rows its index list
// selects, unpacks them on chip, and computes softmax attention with 16-bit
// operands and FP32 accumulation. -1 entries are not loaded.
//
// GB300 design:
//  * Tokens on the UMMA M axis (M = 128 rows per tile), heads on N (16 or 32):
//    S^T[tok, h] = K[tok, :] . q[h, :] and O^T[dim, h] = sum_tok V[tok, dim] P[tok, h].
//  * Rows are gathered by TMA (tile::gather4: four arbitrary 352-byte cache rows
//    per instruction, issued by two producer warps) into a one-tile ring;
//    unusable entries use row -1, which the TMA unit zero-fills.
//  * Eight dequant warps (thread = tile row) convert each row once into the fp16
//    K tile in TMEM (pass A: the A operand of the QK UMMA) and later copy its
//    latent part from TMEM into the V tile in shared memory (pass B: the A
//    operand of PV, read MN-major).
//  * The 576 K columns are split into two halves (latent 0..255 + rope 0..31;
//    latent 256..511 + rope 32..63), each with its own dequant warps, MMA issuer, and
//    barriers, so the halves pipeline independently and meet only in the
//    softmax group (which adds the two partial score accumulators).
//  * Four softmax warps keep a lazily raised running max per head, write P
//    (fp16) to shared memory and accumulate the row sums.
//  * Work is cut stream-K style: the tiles of all (query, head-group) units form
//    one sequence split evenly across the CTAs; each CTA writes one
//    unnormalised partial (O, running max, sum) per unit it touches, and the
//    merge kernel combines them with the log-sum-exp rule.
//  * Operands are FP16: the dequantised e2m1 x E4M3 products are exact in FP16,
//    and q is scaled by a power of two per unit into FP16 range (exact for
//    every element above 2^-24 of the scaled range); the power of two is
//    folded back into the softmax scale.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "decode_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4mla {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kRingStages = 4;            // a tile's rows in 4 quarters of 32 rows, each with its own barrier
// Cache row formats. kFmt 0: the 352-byte NVFP4 row; the ring holds a whole tile (4 buffers of 32
// rows). kFmt 1: the 576-byte FP8 row of the comparison path; kFmt 2: the 672-byte per-token FP8
// row (E4M3 latent / scale, bf16 rope / scale, fp32 scale). For 1 and 2 a whole tile does not fit
// next to the V tile, so the ring holds 2 buffers and quarter q uses buffer q % 2 (quarters 0, 1
// land first, then 2, 3). Rows land densely: gather4 writes 4 rows per instruction, and 4 rows of
// every format are a whole number of 128-byte units (gather destinations must be 128-byte aligned).
// kFmt 2 also keeps the per-row scales of the two tiles in flight (2 x 128 fp32) after the ring.
template <int kFmt>
struct RowFmt {
  static constexpr int kBytes = kFmt == 0 ? kRowBytes : (kFmt == 1 ? kFp8RowBytes : kTokRowBytes);
  static constexpr int kBufs = kFmt == 0 ? 4 : 2;
  static constexpr int kStageBytes = 32 * kBytes;        // 11264 = 88, 18432 = 144, 21504 = 168 x 128 B
  static constexpr int kRingBytes = kBufs * kStageBytes;
  static constexpr int kScaleBytes = kFmt == 2 ? 2 * kTileTokens * 4 : 0;
  static_assert((4 * kBytes) % 128 == 0, "gather4 destinations must stay 128-byte aligned");
};
constexpr int kVBytes = 8 * 128 * 128;    // 8 SW128 atoms x 128 rows x 128 B
constexpr int kTmemCols = 512;
constexpr int kTmemK = 0;                 // K tile: 288 columns (576 fp16 per lane)
constexpr int kTmemS = 288;               // S_a, S_b: NH columns each
// O^T accumulators: 4 M-blocks x NH columns after S_b

struct alignas(16) Smem {
  alignas(16) float m_used[32];      // running max per head (log2 units); read as float4
  alignas(16) float alpha[32];       // rescale factor of this tile per head; read as float4
  uint64_t ring_full[kRingStages];   // gathered rows of a 32-row stage have landed
  uint64_t rows_full[1];             // row numbers + masks of a tile resolved (2 producer warps)
  uint64_t rows_empty[1];            // every stage of that tile has been requested (4 issuing warps)
  // Half h of a tile = latent dims 256h..256h+255 and rope dims 32h..32h+31. Each half has
  // its own dequant warps and MMA issuer, so the two halves pipeline independently and only meet
  // in the softmax.
  // Each issuer commits only where a waiter needs it (a commit costs the issuing thread time):
  // once after its QK, once after its PV.
  uint64_t vfree[2];                 // PV of half h complete: its V rows may be rewritten (1 commit)
  uint64_t kv_ready[2];              // half h of the K tile is in TMEM (4 dequant warps)
  uint64_t s_full;                   // QK of both halves complete (2 commits): S may be read, the K
                                     // tile and the q image rewritten
  uint64_t v_ready[2];               // half h of the V rows of a tile is in shared memory (4 warps)
  uint64_t mask_full[2];             // vmask of a tile written (4 warps), by tile parity
  // P of a tile written and O rescaled (128 threads). One P buffer serves every tile: P(k+1) is
  // written after QK(k+1) completes, which each issuer queued behind its PV(k).
  uint64_t p_full;
  uint64_t o_free;                   // epilogue has read O (128 threads)
  uint64_t q_full[2];                // half h of the unit's q image copied in (issuer h's copy)
  uint64_t drain;                    // every UMMA of both issuers complete
  uint32_t tmem_base;
  volatile int abort;
  alignas(16) int32_t rowbuf[1][kTileTokens];  // producer -> dequant: cache row of every tile entry (-1: unusable)
  uint32_t maskbuf[2][kRingStages];  // producer -> dequant: usable rows of each 32-row stage, by tile parity
  uint32_t stage_cnt[kRingStages];   // dequant warps done with a ring stage (2 per tile)
  uint32_t vmask[2][4];              // dequant -> softmax: usable rows of the tile, by tile parity
  uint32_t maskq[2][4][4];           // folded queries: producer -> dequant, rows of each query token, by tile parity
  uint32_t vmaskq[2][4][4];          // folded queries: dequant -> softmax, rows of each query token
  alignas(16) float red[4][32];      // softmax group: per-warp partial reductions (float4 stores)
  int vote[4];                       // softmax group: does a warp see a score above max + kLazy
  int need_rescale;
  float wmax[12];                    // cluster mode: per-warp |q| maxima of the in-kernel q conversion
};

// Cluster mode, end of the kernel: the partial (m, l) of this CTA and the merge's per-head values,
// kept in the ring buffer (idle once the last tile has been converted).
struct ClusterScratch {
  float cm[32], cl[32];              // this CTA's partial running max and sum per head
  float cw[8][32];                   // weight of each CTA's partial per head
  float cinv[32], clse[32];          // 1 / combined sum, LSE per head
};

// ------------------------------------------------------------------ q image
// q (bf16) of one (query, head group) -> FP16 scaled by 2^e so that max|q| * 2^e lies in
// [2^14, 2^15), written as the exact shared-memory image the decode CTA uses as the UMMA B operand
// (K-major, 128-byte swizzle: 9 atoms of NH rows x 128 B) at dst (global or shared memory).
// Threads tid = 0..kNT-1 take part; the maximum goes through wmax[kNT / 32] and barrier bar
// (0: __syncthreads, else named barrier bar over kNT threads). Every thread returns the unit's
// qscale = softmax_scale * log2(e) * 2^-e. All loads are issued before any is used.
template <int NH, int kNT>
__device__ __forceinline__ float q_image(const DecodeParams& p, int64_t unit, int tid, uint8_t* dst, float* wmax,
                                         int bar) {
  int b, j, hg;
  split_unit(p, unit, b, j, hg);
  const uint16_t* src = p.q + (((int64_t)b * p.Q + j) * p.H + (int64_t)hg * NH) * kQK;
  constexpr int kChunks = NH * (kQK / 8);           // 16-byte chunks of the unit's q block
  constexpr int kPer = (kChunks + kNT - 1) / kNT;
  uint4 v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = tid + kNT * i;
    v[i] = c < kChunks ? __ldg(reinterpret_cast<const uint4*>(src) + c) : make_uint4(0u, 0u, 0u, 0u);
  }
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[t] << 16)), fabsf(__uint_as_float(w[t] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
  if ((tid & 31) == 0) wmax[tid >> 5] = mx;
  if (bar == 0) __syncthreads();
  else asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(kNT) : "memory");
  mx = wmax[0];
#pragma unroll
  for (int i = 1; i < kNT / 32; ++i) mx = fmaxf(mx, wmax[i]);
  int e = 0;
  if (mx > 0.f && isfinite(mx)) {
    int E;
    frexpf(mx, &E);     // mx in [2^(E-1), 2^E)
    e = 15 - E;
  }
  const float up = ldexpf(1.f, e);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int c = tid + kNT * i;
    if (c >= kChunks) break;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const __half2 h = __floats2half2_rn(__uint_as_float(w[t] << 16) * up, __uint_as_float(w[t] & 0xFFFF0000u) * up);
      o[t] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const int h = c / (kQK / 8), cc = c % (kQK / 8);
    const int atom = cc >> 3, ch = cc & 7;
    *reinterpret_cast<uint4*>(dst + atom * (NH * 128) + h * 128 + ((ch ^ (h & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  return p.scale_log2 * ldexpf(1.f, -e);
}

// Refill the ring buffer of quarter q with the 32 rows of tile k (8 gather4 copies, lanes 0..7),
// once the producer has resolved them. Returns false on timeout/abort.
template <int kFmt>
__device__ __forceinline__ bool issue_stage(const DecodeParams& p, Smem* sm, uint8_t* ring, int64_t k, int q, int lane) {
  using F = RowFmt<kFmt>;
  bool good = true;
  if (lane == 0) {
    good = wait(sm, &sm->rows_full[0], (uint32_t)(k & 1), p.status);
    if (good) mbar_arrive_expect_tx(&sm->ring_full[q], (uint32_t)F::kStageBytes);
  }
  good = __shfl_sync(0xffffffffu, good, 0);
  if (!good) return false;
  if (lane < 8) {
    const int4 r = *reinterpret_cast<const int4*>(&sm->rowbuf[0][q * 32 + 4 * lane]);
    gather4(ring + (q % F::kBufs) * F::kStageBytes + lane * 4 * F::kBytes, &p.cache_map, r.x, r.y, r.z, r.w,
            &sm->ring_full[q]);
  }
  __syncwarp();   // every lane has read its row numbers before the table is released
  if (lane == 0) mbar_arrive(&sm->rows_empty[0]);
  return true;
}

// ------------------------------------------------------------------ dequant
// Thread = one tile row (token). Half h: latent dims 256h..256h+255 and rope dims 32h..32h+31.
// FP8 rows: 64 E4M3 bytes -> 32 fp16 pairs (exact). Rows are 576 B apart, so the 16-byte loads of a
// quarter-warp meet four-way bank conflicts; the comparison path keeps the simple layout.
__device__ __forceinline__ void convert_fp8_64(const uint8_t* src, uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r[8 * c + 2 * i] = e4m3x2_to_f16x2(w[i] & 0xFFFFu);
      r[8 * c + 2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
    }
  }
}

// Each dequant warp owns one TMEM lane quarter (tile rows 32q..32q+31) and half of the columns.
// Pass A converts its rows into the fp16 K tile in TMEM (the A operand of the QK UMMA) and then
// releases the ring stage. Pass B copies the latent part of those K rows from TMEM into the
// V tile in shared memory (the A operand of PV, read MN-major) once PV of the previous tile is done
// with those V rows, so the compressed rows are converted only once and leave the ring early.
template <int kFmt, bool kFold>
__device__ void dequant_loop(const DecodeParams& p, Smem* sm, uint8_t* ring, uint8_t* vtile, float* rowscale,
                             int64_t t_begin, int64_t t_end, int warp) {
  using F = RowFmt<kFmt>;
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;               // TMEM lane quarter == tile rows 32q..32q+31
  const int half = (warp - 4) >> 2;
  const int row = 32 * q + lane;
  const uint32_t tmem_row = sm->tmem_base + ((uint32_t)(32 * q) << 16);
  const uint8_t* rowp = ring + (q % F::kBufs) * F::kStageBytes + lane * F::kBytes;
  int64_t n = t_end - t_begin;
  // the last fill this warp requested (quarter, tile); -1: none
  int last_q = -1;
  int64_t last_k = -1;
  // The ring is refilled by the dequant warps themselves: the second of the two warps that read a
  // quarter's buffer issues its next fill as soon as both are done with it (NVFP4: the same
  // quarter of the next tile; FP8: quarter q+2 of this tile, or quarter q-2 of the next). The lo
  // warps issue the first fills.
  if (half == 0 && n > 0 && q < F::kBufs) {
    if (!issue_stage<kFmt>(p, sm, ring, 0, q, lane)) n = 0;
    else last_q = q, last_k = 0;
  }
  for (int64_t g = t_begin; g < t_begin + n; ++g) {
    const int64_t k = g - t_begin;
    // ---- pass A: compressed rows -> fp16 K rows in TMEM
    bool good = true;
    if (lane == 0) {
      good = wait(sm, &sm->ring_full[q], (uint32_t)(k & 1), p.status);
      // the K tile may be rewritten once the previous tile's QK (both halves) is done
      if (good && k > 0) good = wait(sm, &sm->s_full, (uint32_t)((k - 1) & 1), p.status);
    }
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) break;
    __syncwarp();
    tc_fence_after();
    const uint32_t mask = sm->maskbuf[k & 1][q];
    uint32_t r[32];
    if constexpr (kFmt == 0) {
      // the 16 block scales of this half: one 16-byte load instead of four word loads
      const uint4 sc = *reinterpret_cast<const uint4*>(rowp + kScaleOff + 16 * half);
      // Rows of unusable entries arrive zero-filled (scale bytes 0), so they dequantise to zeros.
#pragma unroll 1
      for (int gi = 0; gi < 4; ++gi) {
        const int grp = 4 * half + gi;
        const uint32_t sw = gi == 0 ? sc.x : gi == 1 ? sc.y : gi == 2 ? sc.z : sc.w;
        convert_group(rowp, grp, sw, r);
        __syncwarp();
        tmem_st32(tmem_row + kTmemK + 32 * grp, r);
      }
    } else {
      // FP8 rows: latent byte d is dim d (zero-filled rows give zeros)
#pragma unroll 1
      for (int gi = 0; gi < 4; ++gi) {
        const int grp = 4 * half + gi;
        convert_fp8_64(rowp + 64 * grp, r);
        __syncwarp();
        tmem_st32(tmem_row + kTmemK + 32 * grp, r);
      }
    }
    {
      // rope dims 32 half .. 32 half + 31 -> K columns 256 + 16 half (each half converts 32 of the 64
      // rope dims, so both halves convert 288 dims and issue 18 QK steps)
      uint32_t rr[16];
      if constexpr (kFmt == 2) {
        // bf16 rope / scale -> fp16 (exact for values in fp16's normal range)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + kTokRopeOff + 64 * half + 16 * c);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 h2 = __floats2half2_rn(__uint_as_float(w4[i] << 16), __uint_as_float(w4[i] & 0xFFFF0000u));
            rr[4 * c + i] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
      } else {
        // the rope bytes are E4M3 in both formats
        const uint8_t* src = rowp + (kFmt == 0 ? kRopeOff : kLatent) + 32 * half;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            rr[8 * c + 2 * i] = e4m3x2_to_f16x2(w[i] & 0xFFFFu);
            rr[8 * c + 2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
          }
        }
      }
      __syncwarp();
      tmem_st16(tmem_row + kTmemK + 256 + 16 * half, rr);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if constexpr (kFmt == 2) {
      // the row's scale, for the softmax (published with the row mask)
      if (half == 0) rowscale[(k & 1) * kTileTokens + row] = *reinterpret_cast<const float*>(rowp + kTokScaleOff);
      __syncwarp();
    }
    if constexpr (kFold) {
      if (half == 0 && lane < 4) sm->vmaskq[k & 1][q][lane] = sm->maskq[k & 1][q][lane];
      __syncwarp();
    }
    if (lane == 0) {
      if (half == 0) {
        sm->vmask[k & 1][q] = mask;
        mbar_arrive(&sm->mask_full[k & 1]);
      }
      mbar_arrive(&sm->kv_ready[half]);
    }
    // ---- refill: the second warp done with this quarter's buffer requests its next fill
    {
      uint32_t old = 0;
      if (lane == 0) asm volatile("atom.add.acq_rel.cta.shared::cta.u32 %0, [%1], 1;" : "=r"(old) : "r"(smem_u32(&sm->stage_cnt[q])) : "memory");
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old & 1u) {
        const int nq = F::kBufs == 4 ? q : (q + 2) & 3;
        const int64_t nk = (F::kBufs == 4 || q >= 2) ? k + 1 : k;
        if (nk < n) {
          if (!issue_stage<kFmt>(p, sm, ring, nk, nq, lane)) break;
          last_q = nq, last_k = nk;
        }
      }
    }
    // ---- pass B: latent K rows (TMEM) -> V rows (shared memory, SW128 K-major atoms)
    if (lane == 0) good = wait(sm, &sm->vfree[half], (uint32_t)((k & 1) ^ 1), p.status);
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) break;
    __syncwarp();
    tc_fence_after();
#pragma unroll 1
    for (int gi = 0; gi < 4; ++gi) {
      const int grp = 4 * half + gi;
      tmem_ld32(tmem_row + kTmemK + 32 * grp, r);
      tmem_wait_ld();
      uint8_t* vrow = vtile + grp * 16384 + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(vrow + ((c ^ (row & 7)) << 4)) = make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->v_ready[half]);
  }
  // After an abort, never leave with gathers in flight: wait (bounded) for the last fill this warp
  // requested. (Every earlier fill of the same buffer was waited on before the next one was
  // requested, so the last fills of the warps cover every copy still in flight.)
  if (lane == 0 && last_k >= 0 && sm->abort)
    mbar_wait(&sm->ring_full[last_q], (uint32_t)(last_k & 1), nullptr, kWaitTimeoutNs);
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issue
// Two issuing threads, one per half: issuer h computes the half-h part of QK (K columns of that
// half, into its own S accumulator; the softmax adds the two) and the half-h part of PV (the two
// M-blocks of output dims 256h..256h+255).
template <int NH>
struct MmaIssuer {
  static constexpr uint32_t kIdQK = idesc_f16(128, NH, false, false, false);
  static constexpr uint32_t kIdPV = idesc_f16(128, NH, true, true, false);
  static constexpr uint32_t kPSw = (NH == 32) ? SW_64B : SW_32B;
  static constexpr uint32_t kPSbo = (NH == 32) ? 512 : 256;      // 8 token rows of P
  static constexpr uint32_t kPBytes = 128 * NH * 2;
  const DecodeParams& p;
  Smem* sm;
  int which;
  uint32_t tmem, s_col, o_col;
  uint64_t qd, vd, pd0;
  int64_t t_begin, t_end;
  int64_t ofree_waits = 0;
  uint8_t* q_smem;

  // Copy this half's part of the unit's pre-converted q image (atoms 0..3 for half 0, 4..8 for
  // half 1; issuer 0's QK also reads the rope atom 8, which issuer 1 copies) into the shared q
  // buffer.
  __device__ __forceinline__ void request_q(int64_t unit) {
    const uint32_t atom_bytes = (uint32_t)NH * 128u;
    const uint32_t off = which == 0 ? 0u : 4u * atom_bytes;
    const uint32_t bytes = (which == 0 ? 4u : 5u) * atom_bytes;
    mbar_arrive_expect_tx(&sm->q_full[which], bytes);
    bulk_g2s(q_smem + off, p.q16 + unit * (int64_t)(9u * atom_bytes) + off, bytes, &sm->q_full[which]);
  }

  __device__ __forceinline__ MmaIssuer(const DecodeParams& p_, Smem* sm_, uint8_t* vtile, uint8_t* qs, uint8_t* ps, int64_t tb,
                       int64_t te, int which_)
      : p(p_), sm(sm_), which(which_), t_begin(tb), t_end(te) {
    tmem = sm->tmem_base;
    s_col = tmem + kTmemS + which * NH;
    o_col = tmem + kTmemS + 2 * NH;
    qd = sdesc(smem_u32(qs), 16, 1024, SW_128B);
    q_smem = qs;
    vd = sdesc(smem_u32(vtile), 16384, 1024, SW_128B);
    pd0 = sdesc(smem_u32(ps), 4096, kPSbo, kPSw);
  }

  template <int kAcc>
  __device__ __forceinline__ void qk_step(int ks) {
    umma_ts_w<kAcc>(s_col, tmem + kTmemK + 8 * ks,
                    (uint32_t)qd + (uint32_t)((((ks >> 2) * NH * 128) + (ks & 3) * 32) >> 4), (uint32_t)(qd >> 32),
                    kIdQK);
  }
  __device__ __forceinline__ void qk(int64_t k) {
    tc_fence_after();
    // half h: latent dims 256h..256h+255, then rope dims 32h..32h+31 (K-steps 32 + 2h, 33 + 2h)
    qk_step<0>(16 * which);
#pragma unroll
    for (int x = 1; x < 16; ++x) qk_step<1>(16 * which + x);
    qk_step<1>(32 + 2 * which);
    qk_step<1>(33 + 2 * which);
    umma_commit(&sm->s_full);
  }

  __device__ __forceinline__ void pv(int64_t k, const TileInfo& ti) {
    if (ti.first && k > 0) ++ofree_waits;
    tc_fence_after();
    // P_hi and P_lo planes: the same V rows times each, into the same fp32 accumulator. The half's
    // V rows are released when all of its UMMAs complete (releasing each 32-row chunk as soon as
    // its own UMMAs completed took three more commits per tile and measured slower).
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int mb = which * 2 + mi;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int ks = 2 * w + kk;
          const uint32_t a_lo = (uint32_t)vd + (uint32_t)((mb * 32768 + ks * 2048) >> 4);
          const uint32_t b_lo = (uint32_t)pd0 + (uint32_t)((ks * 2 * kPSbo) >> 4);
          if (ks == 0)
            umma_ss_w<-1>(o_col + mb * NH, a_lo, (uint32_t)(vd >> 32), b_lo, (uint32_t)(pd0 >> 32), kIdPV,
                          ti.first ? 0u : 1u);
          else
            umma_ss_w<1>(o_col + mb * NH, a_lo, (uint32_t)(vd >> 32), b_lo, (uint32_t)(pd0 >> 32), kIdPV);
          umma_ss_w<1>(o_col + mb * NH, a_lo, (uint32_t)(vd >> 32), b_lo + (kPBytes >> 4), (uint32_t)(pd0 >> 32),
                       kIdPV);
        }
      }
    }
    umma_commit(&sm->vfree[which]);
  }
};

// Each issuer runs its half's UMMAs in the pipeline's order QK(0), PV(0), QK(1), PV(1), ..., and
// sleeps in hardware on the barrier it needs next (a polling issuer takes issue slots from the
// warps on its scheduler). PV(k) is ready before QK(k+1): both follow pass B(k) on the dequant
// warps, and QK(k+1) also needs pass A(k+1), which those warps run after pass B(k). When the next
// tile starts a new unit, its q image is requested as soon as QK(k) has completed (the q buffer is
// free then), before the wait for P(k). Every wait below is on a barrier at most one phase ahead
// of the parity it tests (each is released by a step that needs this thread's previous issue).
template <int NH, bool kCluster>
__device__ void mma_loop(const DecodeParams& p, Smem* sm, uint8_t* vtile, uint8_t* qs, uint8_t* ps,
                         int64_t t_begin, int64_t t_end, int which) {
  MmaIssuer<NH> m(p, sm, vtile, qs, ps, t_begin, t_end, which);
  const int64_t n = t_end - t_begin;
  // cluster mode: q_full phase 0 is the unit's q image written in-kernel (no copy to request)
  int64_t q_copies = kCluster ? 1 : 0;
  if (!kCluster && n > 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // q16 comes from the prep grid
    m.request_q(tile_info(p, t_begin, t_begin, t_end).unit);
    q_copies = 1;
  }
  TileInfo ti = tile_info(p, t_begin, t_begin, t_end);
  for (int64_t k = 0; k < n; ++k) {
    // ---- QK(k)
    bool ok = true;
    // issuer 0 also reads the rope atom of the q image, which issuer 1 copies in
    if (ti.first) ok = wait(sm, &sm->q_full[which], (uint32_t)((q_copies - 1) & 1), p.status);
    if (ok && ti.first && which == 0) ok = wait(sm, &sm->q_full[1], (uint32_t)((q_copies - 1) & 1), p.status);
    if (ok) ok = wait(sm, &sm->kv_ready[which], (uint32_t)(k & 1), p.status);
    // (S of tile k-1 has been read: the softmax writes P(k-1) after reading it, and this thread
    // waited for P(k-1) before issuing PV(k-1))
    if (!ok) break;
    m.qk(k);
    TileInfo tn = ti;   // the next tile's info, computed here (off the PV -> QK path)
    if (k + 1 < n) {
      tn = tile_info(p, t_begin + k + 1, t_begin, t_end);
      if (tn.first) {
        // both halves' QK(k) have finished reading the q buffer
        if (!wait(sm, &sm->s_full, (uint32_t)(k & 1), p.status)) break;
        m.request_q(tn.unit);
        ++q_copies;
      }
    }
    // ---- PV(k)
    // the V half is normally in place well before P: test it first, off the P -> PV path
    ok = wait(sm, &sm->v_ready[which], (uint32_t)(k & 1), p.status);
    if (ok) ok = wait(sm, &sm->p_full, (uint32_t)(k & 1), p.status);
    if (ok && ti.first && k > 0) ok = wait(sm, &sm->o_free, (uint32_t)(m.ofree_waits & 1), p.status);
    if (!ok) break;
    m.pv(k, ti);
    ti = tn;
  }
  // never leave with a q copy in flight (abort path)
  if (q_copies > (kCluster ? 1 : 0)) mbar_wait(&sm->q_full[which], (uint32_t)((q_copies - 1) & 1), nullptr, kWaitTimeoutNs);
  // drain: every UMMA of this thread has completed before TMEM is released
  umma_commit(&sm->drain);
  mbar_wait(&sm->drain, 0, nullptr, kWaitTimeoutNs);
}

// ------------------------------------------------------------------ softmax / epilogue
// Scores of this thread's tile row: S = S_a + S_b (the two issuers' halves of the 576-wide
// contraction), loaded one after the other into the same registers; unusable rows become -inf.
template <int NH>
__device__ __forceinline__ void load_scores(uint32_t taddr, bool valid, float qscale, float (&z)[32]) {
  const float kNegInf = __int_as_float(0xff800000);
  uint32_t ra[32];
  __syncwarp();
  if (NH == 32) tmem_ld32(taddr, ra);
  else tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(ra));
  tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 32; ++h) z[h] = h < NH ? __uint_as_float(ra[h]) : 0.f;
  if (NH == 32) tmem_ld32(taddr + NH, ra);
  else tmem_ld16(taddr + NH, *reinterpret_cast<uint32_t(*)[16]>(ra));
  tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 32; ++h) z[h] = (h < NH && valid) ? (z[h] + __uint_as_float(ra[h])) * qscale : kNegInf;
}

// Returns false when the group gave up (abort); every thread of the group returns the same value.
// kFmt 2 (per-token FP8 rows, k = scale_t * k'): the score of row t is scale_t times the UMMA's
// q . k'_t, and PV must weight v'_t by p_t * scale_t. The softmax keeps its reference on the shifted
// exponent z_t + log2(scale_t), so P' = 2^(z_t + log2(scale_t) - m) = p_t * scale_t * 2^-m stays
// inside fp16's range exactly as P does for the other formats, and the row sums add P' / scale_t.
// O and the sums share the reference, so the quotient and the LSE (m + log2 of the sum) are
// unchanged.
template <int NH, bool kCluster, int kFmt = 0, bool kFold = false>
__device__ bool softmax_loop(const DecodeParams& p, Smem* sm, uint8_t* ps, uint8_t* vtile, ClusterScratch* cs,
                             const float* rowscale, int64_t t_begin, int64_t t_end, int64_t cta, float qscale) {
  constexpr uint32_t kPBytes = 128 * NH * 2;
  const int t = threadIdx.x - 384;          // 0..127: tile row / TMEM lane
  const int w = t >> 5, lane = t & 31;
  const uint32_t tmem_lane = sm->tmem_base + ((uint32_t)(32 * w) << 16);
  const uint32_t s_col = kTmemS, o_col = kTmemS + 2 * NH;
  const float kNegInf = __int_as_float(0xff800000);
  float l_part[32];
  bool ok = true;
  if constexpr (!kCluster) asm volatile("griddepcontrol.wait;" ::: "memory");   // qscale comes from the prep kernel
  for (int64_t g = t_begin; g < t_end && ok; ++g) {
    const int64_t k = g - t_begin;
    const TileInfo ti = tile_info(p, g, t_begin, t_end);
    if (ti.first) {
      if constexpr (!kCluster) qscale = p.qscale[ti.unit];
#pragma unroll
      for (int h = 0; h < 32; ++h) l_part[h] = 0.f;
      if (t < 32) sm->m_used[t] = kNegInf;
    }
    // ---- scores of this tile (one waiting thread per warp; the barrier releases the group and
    // agrees on the abort flag)
    if (lane == 0 && wait(sm, &sm->mask_full[k & 1], (uint32_t)((k >> 1) & 1), p.status))
      wait(sm, &sm->s_full, (uint32_t)(k & 1), p.status);
    if (named_sync_softmax_any(sm->abort != 0)) {
      ok = false;
      break;
    }
    tc_fence_after();
    __syncwarp();
    float z[32];
    const bool valid = (sm->vmask[k & 1][w] >> lane) & 1u;
    float inv_rs = 1.f;   // kFmt 2: 1 / scale of this row (0 for an unusable row)
    if constexpr (kFmt == 2) {
      const float rs = rowscale[(k & 1) * kTileTokens + t];
      const bool use = valid && rs > 0.f;
      load_scores<NH>(tmem_lane + s_col, use, qscale * rs, z);
      if (use) {
        const float lrs = __log2f(rs);
#pragma unroll
        for (int h = 0; h < 32; ++h) z[h] += lrs;
        inv_rs = 1.f / rs;
      } else {
        inv_rs = 0.f;
      }
    } else {
      load_scores<NH>(tmem_lane + s_col, valid, qscale, z);
    }
    if constexpr (kFold) {
      // folded queries: column h of head group hg is head (hg * NH + h) % fold_h of query token
      // (hg * NH + h) / fold_h, which uses this row only if the row is in its list and causal range
      int fb, fj, hg;
      split_unit(p, ti.unit, fb, fj, hg);
      uint32_t qb = 0;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) qb |= ((sm->vmaskq[k & 1][w][jj] >> lane) & 1u) << jj;
      const int hshift = __ffs(p.fold_h) - 1;
#pragma unroll
      for (int h = 0; h < NH; ++h)
        if (!((qb >> ((hg * NH + h) >> hshift)) & 1u)) z[h] = kNegInf;
    }
    // ---- lazy running max: vote whether any score exceeds max + kLazy (the first tile of a unit
    // always sets the max, so it skips the vote)
    bool raise = ti.first;
    if (!raise) {
      bool exceed = false;
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        const float4 mv = *reinterpret_cast<const float4*>(&sm->m_used[h]);
        exceed |= (z[h] > mv.x + kLazy) | (z[h + 1] > mv.y + kLazy) | (z[h + 2] > mv.z + kLazy) | (z[h + 3] > mv.w + kLazy);
      }
      const int wv = __any_sync(0xffffffffu, exceed) ? 1 : 0;
      if (lane == 0) sm->vote[w] = wv;
      named_sync_softmax();
      raise = (sm->vote[0] | sm->vote[1] | sm->vote[2] | sm->vote[3]) != 0;
    }
    if (raise) {
      // per-warp maximum of every head over the warp's 32 rows (warp reductions; z stays intact)
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        float4 wm;
        wm.x = redux_max(z[h]);
        wm.y = redux_max(z[h + 1]);
        wm.z = redux_max(z[h + 2]);
        wm.w = redux_max(z[h + 3]);
        if (lane == 0) *reinterpret_cast<float4*>(&sm->red[w][h]) = wm;
      }
      named_sync_softmax();
      if (w == 0) {
        const float tmax = fmaxf(fmaxf(sm->red[0][lane], sm->red[1][lane]), fmaxf(sm->red[2][lane], sm->red[3][lane]));
        const float mold = sm->m_used[lane];
        float mnew = mold, alpha = 1.f;
        if (tmax > mold + kLazy) {
          mnew = tmax;
          alpha = (mold == kNegInf) ? 0.f : ex2_approx(mold - mnew);
        }
        sm->m_used[lane] = mnew;
        sm->alpha[lane] = alpha;
        const bool any = __any_sync(0xffffffffu, lane < NH && alpha != 1.f && mold != kNegInf);
        if (lane == 0) sm->need_rescale = any ? 1 : 0;
      }
      named_sync_softmax();
#pragma unroll
      for (int h = 0; h < 32; h += 4) {
        const float4 av = *reinterpret_cast<const float4*>(&sm->alpha[h]);
        l_part[h] *= av.x; l_part[h + 1] *= av.y; l_part[h + 2] *= av.z; l_part[h + 3] *= av.w;
      }
    }
    tc_fence_before();   // S read (its reuse by the next QK is ordered by the P barrier below)
    // ---- P = 2^(z - m) as two fp16 parts, P_hi = fp16(p) and P_lo = fp16(p - P_hi), rows of the two
    // P planes (MN-major: heads contiguous); PV multiplies V by both and accumulates them in fp32,
    // so the weights carry ~22 bits instead of fp16's 11. (With P_hi alone, the rounding of a few
    // heavy weights moved outputs that cancel to near zero, |out| << sum_t w_t |v_t|, by up to
    // ~90 % of the tolerance on the outlier-heavy keys.) The row sums add the unrounded p.
#pragma unroll
    for (int c = 0; c < NH / 8; ++c) {          // 16-byte chunk c: heads 8c..8c+7
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const int h = 8 * c + i;
        const float m0 = sm->m_used[h], m1 = sm->m_used[h + 1];
        const float p0 = (m0 == kNegInf) ? 0.f : ex2_approx(z[h] - m0);
        const float p1 = (m1 == kNegInf) ? 0.f : ex2_approx(z[h + 1] - m1);
        if constexpr (kFmt == 2) {
          l_part[h] += p0 * inv_rs;
          l_part[h + 1] += p1 * inv_rs;
        } else {
          l_part[h] += p0;
          l_part[h + 1] += p1;
        }
        const __half2 ph = __floats2half2_rn(p0, p1);
        const float2 fh = __half22float2(ph);
        const __half2 pl = __floats2half2_rn(p0 - fh.x, p1 - fh.y);
        hi[i >> 1] = *reinterpret_cast<const uint32_t*>(&ph);
        lo[i >> 1] = *reinterpret_cast<const uint32_t*>(&pl);
      }
      const int off = NH == 32 ? t * 64 + ((c ^ ((t >> 1) & 3)) << 4) : t * 32 + ((c ^ ((t >> 2) & 1)) << 4);
      *reinterpret_cast<uint4*>(ps + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(ps + kPBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();
    // ---- a raised reference: O^T[dim, h] *= alpha[h] before PV(k) adds to it, once PV(k-1) has
    // finished accumulating (P above did not have to wait for this)
    if (raise && sm->need_rescale && !ti.first) {
      if (lane == 0 && wait(sm, &sm->vfree[0], (uint32_t)((k - 1) & 1), p.status))
        wait(sm, &sm->vfree[1], (uint32_t)((k - 1) & 1), p.status);
      __syncwarp();
      tc_fence_after();
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        uint32_t r[32];
        if (NH == 32) {
          tmem_ld32(tmem_lane + o_col + mb * NH, r);
        } else {
          tmem_ld16(tmem_lane + o_col + mb * NH, *reinterpret_cast<uint32_t(*)[16]>(r));
        }
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < NH; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * sm->alpha[h]);
        if (NH == 32) tmem_st32(tmem_lane + o_col + mb * NH, r);
        else tmem_st16(tmem_lane + o_col + mb * NH, *reinterpret_cast<uint32_t(*)[16]>(r));
      }
      tmem_wait_st();
      tc_fence_before();
    }
    mbar_arrive(&sm->p_full);

    if (ti.last) {
      // ---- epilogue: write this segment's unnormalised partial
      // O is final once both halves' PV of this tile has completed
      if (lane == 0 && wait(sm, &sm->vfree[0], (uint32_t)(k & 1), p.status))
        wait(sm, &sm->vfree[1], (uint32_t)(k & 1), p.status);
      if (named_sync_softmax_any(sm->abort != 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t slot = cta + ti.unit;
      // stream-K: partial to the workspace; cluster mode: to this CTA's V tile (free now: the last
      // PV is complete), read by the cluster's CTAs through distributed shared memory
      float* po = kCluster ? reinterpret_cast<float*>(vtile) : p.part_o + slot * (int64_t)NH * kLatent;
      {
        float v[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) v[h] = l_part[h];
        const float ws = warp_transpose_reduce<1>(v);
        sm->red[w][lane] = ws;
      }
      named_sync_softmax();
      if (t < NH) {
        const float lsum = sm->red[0][t] + sm->red[1][t] + sm->red[2][t] + sm->red[3][t];
        if constexpr (kCluster) {
          cs->cm[t] = sm->m_used[t];
          cs->cl[t] = lsum;
        } else {
          p.part_ml[(slot * NH + t) * 2 + 0] = sm->m_used[t];
          p.part_ml[(slot * NH + t) * 2 + 1] = lsum;
        }
      }
      __syncwarp();
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        uint32_t r[32];
        if (NH == 32) {
          tmem_ld32(tmem_lane + o_col + mb * NH, r);
        } else {
          tmem_ld16(tmem_lane + o_col + mb * NH, *reinterpret_cast<uint32_t(*)[16]>(r));
        }
        tmem_wait_ld();
        const int dim = mb * 128 + t;
#pragma unroll
        for (int h = 0; h < NH; ++h) po[(int64_t)h * kLatent + dim] = __uint_as_float(r[h]);
      }
      tc_fence_before();
      mbar_arrive(&sm->o_free);
      named_sync_softmax();
    }
  }
  return ok;
}

// ------------------------------------------------------------------ cluster merge
// Cluster mode: the G CTAs of a cluster hold the partials (O [NH][512] fp32 in their V tiles,
// running max m and sum l per head) of one unit. CTA r combines latent dims [512r/G, 512(r+1)/G)
// (rounded to 64) of every head with the log-sum-exp rule (m* = max m_g, w_g = 2^(m_g - m*),
// O = sum w_g O_g / sum w_g l_g), reading the other CTAs' partials through distributed shared
// memory, and writes the bf16 output; CTA 0 writes the LSE (natural log).
template <int NH>
__device__ void cluster_merge(const DecodeParams& p, ClusterScratch* sm, uint8_t* vtile, int64_t unit, int rank,
                              bool have) {
  const int G = p.cluster;
  const float kNegInf = __int_as_float(0xff800000);
  if (!have && threadIdx.x < NH) {   // no tiles here: contribute nothing
    sm->cm[threadIdx.x] = kNegInf;
    sm->cl[threadIdx.x] = 0.f;
  }
  cluster_sync_all();
  if (threadIdx.x < NH) {
    const int h = threadIdx.x;
    const uint32_t am = smem_u32(&sm->cm[h]), al = smem_u32(&sm->cl[h]);
    float m[8], l[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      m[g] = g < G ? ld_dsmem_f32(map_shared_rank(am, (uint32_t)g)) : kNegInf;
      l[g] = g < G ? ld_dsmem_f32(map_shared_rank(al, (uint32_t)g)) : 0.f;
    }
    float mstar = kNegInf;
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (l[g] > 0.f) mstar = fmaxf(mstar, m[g]);
    float lsum = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const float w = l[g] > 0.f ? exp2f(m[g] - mstar) : 0.f;
      lsum += w * l[g];
      sm->cw[g][h] = w;
    }
    sm->cinv[h] = lsum > 0.f ? 1.f / lsum : 0.f;
    sm->clse[h] = lsum > 0.f ? (mstar + log2f(lsum)) * 0.69314718055994530942f : kNegInf;
  }
  __syncthreads();
  int b, j, hg;
  split_unit(p, unit, b, j, hg);
  const int64_t row0 = ((int64_t)b * p.Q + j) * p.H + (int64_t)hg * NH;
  if (rank == 0 && threadIdx.x < NH) p.lse[row0 + threadIdx.x] = sm->clse[threadIdx.x];
  const int d_lo = (kLatent / 8) * ((rank * 8) / G), d_hi = (kLatent / 8) * (((rank + 1) * 8) / G);
  const int span4 = (d_hi - d_lo) / 4;   // float4 items per head
  const int total = NH * span4;
  const uint32_t base = smem_u32(vtile);
  constexpr int kBatch = 4;   // items per thread per round; every CTA's loads for them are issued together
  for (int it0 = threadIdx.x; it0 < total; it0 += kThreads * kBatch) {
    int hh[kBatch], dd[kBatch];
    float4 acc[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int it = it0 + i * kThreads;
      hh[i] = it < total ? it / span4 : 0;
      dd[i] = it < total ? d_lo + 4 * (it - hh[i] * span4) : d_lo;
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int g = 0; g < G; ++g) {
      float4 o[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        o[i] = ld_dsmem_f4(map_shared_rank(base + (uint32_t)(hh[i] * kLatent + dd[i]) * 4u, (uint32_t)g));
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const float w = sm->cw[g][hh[i]];
        acc[i].x += w * o[i].x;
        acc[i].y += w * o[i].y;
        acc[i].z += w * o[i].z;
        acc[i].w += w * o[i].w;
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (it0 + i * kThreads >= total) break;
      const float inv = sm->cinv[hh[i]];
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
      uint2 packed;
      packed.x = *reinterpret_cast<const uint32_t*>(&lo);
      packed.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(p.out + (row0 + hh[i]) * kLatent + dd[i]) = packed;
    }
  }
  // no CTA leaves (and releases its shared memory) while another may still read it
  cluster_sync_all();
}

// kCluster: the cluster schedule (in-kernel q, DSMEM merge). kPublish: the split schedule with a
// polling merge grid (results in host memory): each CTA tags its partial slots when done. The
// tagging is a separate instance because its mere presence slowed the other split kernel by ~2 %.
template <int NH, bool kCluster, bool kPublish, int kFmt = 0, bool kFold = false>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(kFmt == 0 || !kCluster, "FP8 rows run on the split schedule only");
  static_assert(!kFold || (!kCluster && !kPublish && kFmt == 0),
                "folded queries run on the split schedule with results in device memory");
  static_assert(kFmt == 0 || !kPublish, "FP8 rows write their results to device memory only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* vtile = base;                                   // 131072
  uint8_t* qs = vtile + kVBytes;                           // 9 * NH * 128
  uint8_t* ps = qs + 9 * NH * 128;                         // 2 x 128 * NH * 2 (P, double-buffered)
  uint8_t* ring = ps + 2 * 128 * NH * 2;                   // RowFmt<kFmt>::kRingBytes
  static_assert(RowFmt<kFmt>::kRingBytes % 16 == 0, "control block must stay 16-byte aligned");
  float* rowscale = reinterpret_cast<float*>(ring + RowFmt<kFmt>::kRingBytes);   // kFmt 2 only
  Smem* sm = reinterpret_cast<Smem*>(ring + RowFmt<kFmt>::kRingBytes + RowFmt<kFmt>::kScaleBytes);

  const int warp = threadIdx.x >> 5;
  const int64_t cta = blockIdx.x;
  int64_t t_begin, t_end;
  if constexpr (kCluster) {
    // cluster u (CTAs uG .. uG+G-1) owns unit u; CTA rank r takes the r-th share of its tiles
    const int64_t unit = cta / p.cluster, r = cta % p.cluster;
    t_begin = unit * p.tiles_per_unit + r * p.tiles_per_unit / p.cluster;
    t_end = unit * p.tiles_per_unit + (r + 1) * p.tiles_per_unit / p.cluster;
  } else {
    // Every decode CTA is resident once all of them reach this point, so letting the
    // merge grid be scheduled now cannot take resources a decode CTA still needs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    t_begin = range_begin(p, cta);
    t_end = range_begin(p, cta + 1);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingStages; ++i) {
      mbar_init(&sm->ring_full[i], 1);
      sm->stage_cnt[i] = 0;
    }
    mbar_init(&sm->rows_full[0], 2);
    mbar_init(&sm->rows_empty[0], 4);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sm->vfree[h], 1);
      mbar_init(&sm->kv_ready[h], 4);
      mbar_init(&sm->v_ready[h], 4);
      mbar_init(&sm->mask_full[h], 4);
    }
    mbar_init(&sm->s_full, 2);
    mbar_init(&sm->p_full, 128);
    mbar_init(&sm->o_free, 128);
    mbar_init(&sm->q_full[0], kCluster ? 384 : 1);   // cluster mode: the converting threads
    mbar_init(&sm->q_full[1], kCluster ? 384 : 1);
    mbar_init(&sm->drain, 2);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  float qscale = 0.f;
  if constexpr (kCluster) {
    // The dequant and softmax warps (idle until the first tile arrives) write the unit's q image
    // straight into the q buffer; the UMMAs read it through the async proxy once every writer
    // has arrived on q_full.
    if (warp >= 4) {
      qscale = q_image<NH, 384>(p, cta / p.cluster, threadIdx.x - 128, qs, sm->wmax, 2);
      fence_proxy_async_smem();
      mbar_arrive(&sm->q_full[0]);
      mbar_arrive(&sm->q_full[1]);
    }
  }
  if (warp == 0 || warp == 3) {
    producer_loop<kFold, 2, 1>(p, sm, t_begin, t_end, warp == 0 ? 0 : 1);
  } else if (warp == 1 || warp == 2) {
    if ((threadIdx.x & 31) == 0) mma_loop<NH, kCluster>(p, sm, vtile, qs, ps, t_begin, t_end, warp - 1);
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    dequant_loop<kFmt, kFold>(p, sm, ring, vtile, rowscale, t_begin, t_end, warp);
  } else if (warp >= 12) {
    const bool ok = softmax_loop<NH, kCluster, kFmt, kFold>(p, sm, ps, vtile, reinterpret_cast<ClusterScratch*>(ring),
                                                     rowscale, t_begin, t_end, cta, qscale);
    if constexpr (kPublish) {
      // Polling merge (results in host memory): publish this CTA's partials. Every writer fences
      // its stores at GPU scope, then one thread tags the CTA's slots, which the merge grid polls
      // instead of waiting for the whole decode grid.
      if (ok && t_begin < t_end) {
        __threadfence();
        named_sync_softmax();
        if (threadIdx.x == 384) {
          const int64_t u0 = t_begin / p.tiles_per_unit, u1 = (t_end - 1) / p.tiles_per_unit;
          for (int64_t u = u0; u <= u1; ++u) st_relaxed_gpu_u64(p.part_flag + cta + u, p.tag);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(sm->tmem_base, kTmemCols);
  }
  if constexpr (kCluster)
    cluster_merge<NH>(p, reinterpret_cast<ClusterScratch*>(ring), vtile, cta / p.cluster, (int)(cta % p.cluster),
                      t_begin < t_end);
}

// ------------------------------------------------------------------ q prep
// Stream-K mode: each 256-thread group of a block writes one (query, head group) unit's FP16 q
// image (see q_image) and its qscale to the workspace, for the decode CTAs to copy. Two units per
// block: a decode CTA cannot share an SM with a prep block, so the fewer SMs the prep grid holds,
// the fewer decode CTAs start late (those get the shorter stream-K shares).
constexpr int kPrepUnitsPerBlock = 2;
template <int NH>
__global__ void __launch_bounds__(256 * kPrepUnitsPerBlock) q_prep_kernel(const DecodeParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float wmax[kPrepUnitsPerBlock][8];
  const int grp = threadIdx.x >> 8, tid = threadIdx.x & 255;
  const int64_t unit = (int64_t)blockIdx.x * kPrepUnitsPerBlock + grp;
  if (unit >= p.units) return;   // a whole group (its named barrier is its own)
  int b, j, hg;
  split_unit(p, unit, b, j, hg);
  if (hg == 0) {
    // Warm L2 with this query's index list and (once per request) the request's page-table row:
    // the decode grid resolves its first tiles from them while this grid runs.
    const char* tk = reinterpret_cast<const char*>(p.idx + ((int64_t)b * p.Q + j) * p.topk);
    const int64_t tk_bytes = (int64_t)p.topk * 4;
    for (int64_t o = (int64_t)tid * 128; o < tk_bytes; o += 256 * 128) prefetch_l2(tk + o);
    if (j == 0) {
      const char* pt = reinterpret_cast<const char*>(p.page_table + (int64_t)b * p.max_pages);
      const int64_t pt_bytes = p.max_pages * 4;
      for (int64_t o = (int64_t)tid * 128; o < pt_bytes; o += 256 * 128) prefetch_l2(pt + o);
    }
  }
  const float qscale = q_image<NH, 256>(p, unit, tid, p.q16 + unit * (int64_t)(9 * NH * 128), wmax[grp], 1 + grp);
  if (tid == 0) p.qscale[unit] = qscale;
}

// ------------------------------------------------------------------ merge
// Block (virtual unit, group of 8 heads), 512 threads: 64 threads per head, 8 latent dims each.
// Combines the partials of the CTAs that covered the
// unit with the log-sum-exp rule (m* = max m_s, w_s = 2^(m_s - m*), O = sum w_s O_s / sum w_s l_s);
// writes bf16 out and fp32 LSE (natural log). For units covered by up to kMax CTAs every load is
// issued before any is used (one memory round trip). The grid is launched early (programmatic
// dependent launch). When out and LSE live in host memory (merge_poll), each block starts as soon
// as its unit's partials are tagged, so most of the results cross the host link while the last
// decode CTAs still run; otherwise the block waits for the decode grid, which costs less than
// the tags' fences when the results stay on the device.
constexpr int kMergeThreads = 128;   // 64 threads per head; small blocks keep the grid in one wave

// Partial loads: L2 only when polling (a slot is rewritten by every call, and only thread 0 of the
// block performed the acquire); plain loads after the grid-completion wait.
template <bool kPoll, class T>
__device__ __forceinline__ T ld_partial(const T* ptr) {
  if constexpr (kPoll) return __ldcg(ptr);
  else return *ptr;
}

// Fold partial slots base .. base+3 (those below n) of one (unit, head) into the running
// (max, sum, O) of the merge: max and sum in log2 units, O unnormalised.
constexpr int kMergeChunk = 4;
template <int NH, bool kPoll>
__device__ __forceinline__ void merge_chunk(const float2* ml_base, const float4* o_base, int base, int n, float& mstar,
                                            float& lsum, float4& a0, float4& a1) {
  constexpr int64_t kSlotO = (int64_t)NH * kLatent / 4;   // float4 stride between slots
  const float kNegInf = __int_as_float(0xff800000);
  float2 ml[kMergeChunk];
  float4 o0[kMergeChunk], o1[kMergeChunk];
#pragma unroll
  for (int i = 0; i < kMergeChunk; ++i) {
    const bool in = base + i < n;
    const int64_t s = base + i;
    ml[i] = in ? ld_partial<kPoll>(ml_base + s * NH) : make_float2(kNegInf, 0.f);
    o0[i] = in ? ld_partial<kPoll>(o_base + s * kSlotO) : make_float4(0.f, 0.f, 0.f, 0.f);
    o1[i] = in ? ld_partial<kPoll>(o_base + s * kSlotO + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float cmax = kNegInf;
#pragma unroll
  for (int i = 0; i < kMergeChunk; ++i)
    if (ml[i].y > 0.f) cmax = fmaxf(cmax, ml[i].x);
  if (cmax == kNegInf) return;
  if (cmax > mstar) {
    if (mstar != kNegInf) {
      const float r = exp2f(mstar - cmax);
      lsum *= r;
      a0.x *= r; a0.y *= r; a0.z *= r; a0.w *= r;
      a1.x *= r; a1.y *= r; a1.z *= r; a1.w *= r;
    }
    mstar = cmax;
  }
#pragma unroll
  for (int i = 0; i < kMergeChunk; ++i) {
    if (!(ml[i].y > 0.f)) continue;
    const float w = exp2f(ml[i].x - mstar);
    lsum += w * ml[i].y;
    a0.x += w * o0[i].x; a0.y += w * o0[i].y; a0.z += w * o0[i].z; a0.w += w * o0[i].w;
    a1.x += w * o1[i].x; a1.y += w * o1[i].y; a1.z += w * o1[i].z; a1.w += w * o1[i].w;
  }
}

template <int NH, bool kPoll>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p) {
  if constexpr (!kPoll) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t unit = blockIdx.x;
  const int h = blockIdx.y * (kMergeThreads / 64) + (threadIdx.x >> 6);
  const int d8 = threadIdx.x & 63;                 // dims 8*d8 .. 8*d8+7
  const int64_t g0 = unit * p.tiles_per_unit, g1 = g0 + p.tiles_per_unit - 1;
  const int64_t c_lo = range_of_tile(p, g0);
  const int64_t c_hi = range_of_tile(p, g1);
  const int n = (int)(c_hi - c_lo + 1);   // CTAs (partial slots) that covered the unit
  const float kNegInf = __int_as_float(0xff800000);
  if constexpr (kPoll) {
    // Polling mode: the unit's partials are complete once every covering CTA has tagged its slot
    // with this call's tag (bounded wait; the barrier passes thread 0's acquire on to the block).
    __shared__ int ready;
    if (threadIdx.x == 0) {
      bool ok = true;
      uint64_t t0 = 0;
      for (int i = 0; i < n && ok; ++i) {
        const uint64_t* f = p.part_flag + c_lo + unit + i;
        for (uint32_t it = 0; ld_acquire_gpu_u64(f) != p.tag; ++it) {
          __nanosleep(128);
          if ((it & 63u) == 63u) {
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitTimeoutNs) {
              ok = false;
              break;
            }
          }
        }
      }
      if (!ok && p.status != nullptr) atomicAdd(p.status + 2, 1);
      ready = ok ? 1 : 0;
    }
    __syncthreads();
    if (!ready) return;
  }
  const float2* ml_base = reinterpret_cast<const float2*>(p.part_ml) + (c_lo + unit) * NH + h;
  const float4* o_base = reinterpret_cast<const float4*>(p.part_o + ((c_lo + unit) * NH + h) * (int64_t)kLatent) + 2 * d8;
  float mstar = kNegInf, lsum = 0.f;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  // Slots in chunks of four, every load of a chunk issued before any is used; the running sums are
  // rescaled when a later chunk raises the maximum, so a unit split over many CTAs costs one L2
  // round trip per chunk instead of one per slot. (One chunk, the usual case, is its own copy:
  // with the chunk base fixed at 0 the loads and their predicates are set up ahead.)
  if (n <= kMergeChunk) merge_chunk<NH, kPoll>(ml_base, o_base, 0, n, mstar, lsum, a0, a1);
  else
    for (int base = 0; base < n; base += kMergeChunk) merge_chunk<NH, kPoll>(ml_base, o_base, base, n, mstar, lsum, a0, a1);
  int b, j, hg;
  split_unit(p, unit, b, j, hg);
  const int64_t row = ((int64_t)b * p.Q + j) * p.H + (int64_t)hg * NH + h;
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  const __nv_bfloat162 v0 = __floats2bfloat162_rn(a0.x * inv, a0.y * inv);
  const __nv_bfloat162 v1 = __floats2bfloat162_rn(a0.z * inv, a0.w * inv);
  const __nv_bfloat162 v2 = __floats2bfloat162_rn(a1.x * inv, a1.y * inv);
  const __nv_bfloat162 v3 = __floats2bfloat162_rn(a1.z * inv, a1.w * inv);
  reinterpret_cast<uint4*>(p.out + row * kLatent)[d8] =
      make_uint4(*reinterpret_cast<const uint32_t*>(&v0), *reinterpret_cast<const uint32_t*>(&v1),
                 *reinterpret_cast<const uint32_t*>(&v2), *reinterpret_cast<const uint32_t*>(&v3));
  if (d8 == 0) p.lse[row] = lsum > 0.f ? (mstar + log2f(lsum)) * 0.69314718055994530942f : kNegInf;
}

template <int NH, int kFmt = 0>
constexpr size_t decode_smem_bytes() {
  return 1024 + kVBytes + 9 * NH * 128 + 2 * 128 * NH * 2 + RowFmt<kFmt>::kRingBytes + RowFmt<kFmt>::kScaleBytes +
         sizeof(Smem);
}
static_assert(decode_smem_bytes<32>() <= 232448, "decode CTA exceeds the 227 KB shared-memory limit");
static_assert(decode_smem_bytes<32, 1>() <= 232448, "FP8 decode CTA exceeds the 227 KB shared-memory limit");
static_assert(decode_smem_bytes<32, 2>() <= 232448, "per-token FP8 decode CTA exceeds the 227 KB shared-memory limit");
static_assert(sizeof(ClusterScratch) <= RowFmt<0>::kRingBytes, "cluster scratch lives in the ring");

}  // namespace

static cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Kernel attributes are set once per device (a cudaFuncSetAttribute between the prep launch and the
// decode launch would keep the decode grid from starting while the prep grid runs).
static cudaError_t set_attributes() {
  cudaError_t result = cudaSuccess;
  const void* small[6] = {(const void*)q_prep_kernel<32>,        (const void*)q_prep_kernel<16>,
                          (const void*)merge_kernel<32, false>, (const void*)merge_kernel<16, false>,
                          (const void*)merge_kernel<32, true>,  (const void*)merge_kernel<16, true>};
  // The prep and merge grids ask for the same (maximum) shared-memory carveout as the decode grid,
  // so an SM does not have to be reconfigured between the three kernels.
  for (const void* f : small) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess && result == cudaSuccess) result = e;
  }
  const void* big[12] = {(const void*)decode_kernel<32, false, false>,    (const void*)decode_kernel<32, false, true>,
                         (const void*)decode_kernel<32, true, false>,     (const void*)decode_kernel<16, false, false>,
                         (const void*)decode_kernel<16, false, true>,     (const void*)decode_kernel<16, true, false>,
                         (const void*)decode_kernel<32, false, false, 1>, (const void*)decode_kernel<16, false, false, 1>,
                         (const void*)decode_kernel<32, false, false, 2>, (const void*)decode_kernel<16, false, false, 2>,
                         (const void*)decode_kernel<32, false, false, 0, true>,
                         (const void*)decode_kernel<16, false, false, 0, true>};
  const int bytes[12] = {(int)decode_smem_bytes<32>(),    (int)decode_smem_bytes<32>(), (int)decode_smem_bytes<32>(),
                         (int)decode_smem_bytes<16>(),    (int)decode_smem_bytes<16>(), (int)decode_smem_bytes<16>(),
                         (int)decode_smem_bytes<32, 1>(), (int)decode_smem_bytes<16, 1>(),
                         (int)decode_smem_bytes<32, 2>(), (int)decode_smem_bytes<16, 2>(),
                         (int)decode_smem_bytes<32>(),    (int)decode_smem_bytes<16>()};
  static_assert(sizeof(big) / sizeof(big[0]) == sizeof(bytes) / sizeof(bytes[0]), "one size per decode instance");
  for (int i = 0; i < 12; ++i) {
    const cudaError_t e = cudaFuncSetAttribute(big[i], cudaFuncAttributeMaxDynamicSharedMemorySize, bytes[i]);
    if (e != cudaSuccess && result == cudaSuccess) result = e;
  }
  return result;
}

static cudaError_t set_attributes_once() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return set_attributes();
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  err = set_attributes();
  if (err == cudaSuccess) done[dev] = true;
  return err;
}

static cudaLaunchAttribute cluster_attr(int g) {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = (unsigned)g;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// Stream-K: q prep (ordinary launch) -> decode (PDL) -> merge (PDL): each dependent grid is
// launched early and waits with griddepcontrol.wait before reading its inputs. The pair schedule
// runs the same three grids with the pair decode grid in the middle.
// Cluster mode: the decode grid alone (q converted in-kernel, partials merged on chip).
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t err = set_attributes_once();
  if (err != cudaSuccess) return err;
  const bool h32 = p.heads_per_cta == 32;
  if (p.cluster > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = h32 ? decode_smem_bytes<32>() : decode_smem_bytes<16>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {cluster_attr(p.cluster)};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (h32) return cudaLaunchKernelEx(&cfg, decode_kernel<32, true, false>, p);
    return cudaLaunchKernelEx(&cfg, decode_kernel<16, true, false>, p);
  }
  const unsigned prep_blocks = (unsigned)((p.units + kPrepUnitsPerBlock - 1) / kPrepUnitsPerBlock);
  if (h32) q_prep_kernel<32><<<prep_blocks, 256 * kPrepUnitsPerBlock, 0, stream>>>(p);
  else q_prep_kernel<16><<<prep_blocks, 256 * kPrepUnitsPerBlock, 0, stream>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (p.pair) return launch_decode_pair(p, stream);   // decode_pair.cu
  const size_t smem = p.row_fmt == 1   ? (h32 ? decode_smem_bytes<32, 1>() : decode_smem_bytes<16, 1>())
                     : p.row_fmt == 2 ? (h32 ? decode_smem_bytes<32, 2>() : decode_smem_bytes<16, 2>())
                                      : (h32 ? decode_smem_bytes<32>() : decode_smem_bytes<16>());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.row_fmt == 1) {   // FP8 rows: results in device memory (the host checks)
    if (h32) return cudaLaunchKernelEx(&cfg, decode_kernel<32, false, false, 1>, p);
    return cudaLaunchKernelEx(&cfg, decode_kernel<16, false, false, 1>, p);
  }
  if (p.fold_q > 1) {     // folded queries: results in device memory (the host checks)
    if (h32) return cudaLaunchKernelEx(&cfg, decode_kernel<32, false, false, 0, true>, p);
    return cudaLaunchKernelEx(&cfg, decode_kernel<16, false, false, 0, true>, p);
  }
  if (p.row_fmt == 2) {   // per-token FP8 rows: results in device memory (the host checks)
    if (h32) return cudaLaunchKernelEx(&cfg, decode_kernel<32, false, false, 2>, p);
    return cudaLaunchKernelEx(&cfg, decode_kernel<16, false, false, 2>, p);
  }
  if (p.merge_poll) {
    if (h32) return cudaLaunchKernelEx(&cfg, decode_kernel<32, false, true>, p);
    return cudaLaunchKernelEx(&cfg, decode_kernel<16, false, true>, p);
  }
  if (h32) return cudaLaunchKernelEx(&cfg, decode_kernel<32, false, false>, p);
  return cudaLaunchKernelEx(&cfg, decode_kernel<16, false, false>, p);
}

int max_active_clusters(int heads_per_cta, int cluster) {
  if (set_attributes_once() != cudaSuccess) return 0;
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int cache[kMaxDevices][2][9] = {};   // value + 1; 0 = not computed yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cluster < 1 || cluster > 8) return 0;
  const int hi = heads_per_cta == 32 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDevices && cache[dev][hi][cluster] > 0) return cache[dev][hi][cluster] - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cluster * 64), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = hi ? decode_smem_bytes<32>() : decode_smem_bytes<16>();
  cudaLaunchAttribute attr[1] = {cluster_attr(cluster)};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = hi ? cudaOccupancyMaxActiveClusters(&n, decode_kernel<32, true, false>, &cfg)
                           : cudaOccupancyMaxActiveClusters(&n, decode_kernel<16, true, false>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev][hi][cluster] = n + 1;
  return n;
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.units, (unsigned)(p.heads_per_cta / (kMergeThreads / 64)), 1);
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.merge_poll) {
    if (p.heads_per_cta == 32) return cudaLaunchKernelEx(&cfg, merge_kernel<32, true>, p);
    return cudaLaunchKernelEx(&cfg, merge_kernel<16, true>, p);
  }
  if (p.heads_per_cta == 32) return cudaLaunchKernelEx(&cfg, merge_kernel<32, false>, p);
  return cudaLaunchKernelEx(&cfg, merge_kernel<16, false>, p);
}

}  // namespace nvfp4mla
