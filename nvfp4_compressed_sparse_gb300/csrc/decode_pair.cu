// Pair decode kernel: the split decode with the two halves of the 576-wide contraction placed in the
// two CTAs of a 2-CTA thread-block cluster instead of one CTA.
//
// What is computed is exactly what the split kernel (decode_kernel.cu) computes ("Prime Inference",
// translated page, "Native NVFP4 sparse MLA decode kernel"): per (query, head group) unit, the
// softmax attention of the query's heads over the cache rows its index list selects, unpacked on
// chip, with FP16 operands and FP32 accumulation, cut stream-K into partials that the merge grid
// combines. The scores, maxima, P and sums are the split kernel's bit for bit; the one difference is
// that PV accumulates V.P_hi and V.P_lo in two fp32 accumulators added at the end instead of one
// (a different rounding order of the same fp32 sums).
//
// Why two CTAs: in one CTA the fp16 K tile (288 TMEM columns), the V tile (128 KB of shared memory)
// and the one-tile ring of gathered rows fill TMEM and shared memory, so every buffer is single and
// the stages of consecutive tiles wait on each other. CTA h of a pair holds only half h (latent dims
// 256h..256h+255 and rope dims 32h..32h+31): half the K tile, half the V tile, half the q image and
// half of the O accumulator. The room this frees double-buffers K and S in TMEM and deepens the ring
// to two tiles, and leaves the TMEM for a PV of N = 2 NH. The price is one exchange per tile: the
// two partial score tiles (QK over each half) are added in both CTAs, each sending its 128 x NH fp32
// partial to the other through distributed shared memory, and both CTAs run the (identical) softmax.
//
// Roles per CTA (20 warps): 0, 3 producers (row resolution, as in the split kernel); 1 and 2 MMA
// issuers (QK, PV); 4..11 dequant (lane quarter q = warp & 3, sub-half s: two of the half's four 64-dim groups and
// 32 of its rope dims); 12..19 softmax and epilogue (two warps per lane quarter, half the heads each). Every wait is bounded (2 s); a CTA that gives
// up sets its abort flag, and its partner gives up on its own bounded waits, so both always reach
// the closing cluster barrier.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "decode_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4mla {
namespace {

using namespace ptx;

constexpr int kPairThreads = 640;
constexpr int kPairStages = 8;                          // ring: two tiles x four 32-row quarters
constexpr int kPairStageBytes = 32 * kRowBytes;         // 11264 (88 x 128 B)
constexpr int kPairRingBytes = kPairStages * kPairStageBytes;
constexpr int kPairVBytes = 4 * 128 * 128;              // the half's 256 latent dims: 4 SW128 atoms x 128 rows
constexpr int kPairQAtoms = 5;                          // q image atoms of a half: its 4 latent atoms + the rope atom
constexpr int kPairKCols = 160;                         // one K buffer: 128 latent + 16 rope columns (+ 16 spare)
constexpr int kPairTmemS = 2 * kPairKCols;              // two S buffers (NH columns each), then O^T: 2 M-blocks
                                                        // of [O_hi | O_lo] (2 NH columns each)
constexpr uint32_t kPairTmemCols = 512;

struct alignas(16) PairSmem {
  alignas(16) float m_used[32];      // running max per head (log2 units); read as float4
  alignas(16) float alpha[32];       // rescale factor of this tile per head
  uint64_t ring_full[kPairStages];   // stage (tile parity, quarter): its 32 gathered rows have landed
  uint64_t rows_full[2];             // row numbers + masks of tile k resolved (2 producer warps), table k % 2
  uint64_t rows_empty[2];            // every stage of the table's tile has been requested (4 requests)
  uint64_t kv_ready[2];              // K buffer b holds its tile (8 dequant warps)
  uint64_t qk_done[2];               // QK of the tile in K buffer b complete: K buffer b and S buffer b
  uint64_t s_free[2];                // softmax has read S buffer b (8 warps)
  uint64_t mask_full[4];             // vmask of tile k written (4 warps), entry k % 4
  uint64_t v_ready;                  // V rows of a tile in shared memory (8 dequant warps)
  uint64_t vfree[4];                 // PV has finished reading V rows 32w..32w+31 (and, for w = 3, P)
  uint64_t p_full;                   // P of a tile written and O rescaled (256 softmax threads)
  uint64_t o_done;                   // last PV of a unit segment complete
  uint64_t o_free;                   // epilogue has read O (256 softmax threads)
  uint64_t q_full;                   // the unit's q image (this half's atoms) copied in
  uint64_t x_full[2];                // the partner's partial scores of tile k are in xbuf[k % 2] (this CTA's
                                     // expect-tx arrival + the bytes of the partner's asynchronous stores)
  uint64_t x_free[2];                // the partner has read what this CTA sent into its xbuf[b] (8 remote warps)
  uint64_t drain;                    // every UMMA of both issuers complete
  uint32_t tmem_base;
  volatile int abort;
  // producer -> dequant: cache row of every entry of tile k (-1: unusable), table k % 2. The ring runs
  // two tiles ahead of the conversion, so a refill request for tile k+2 can come before tile k+1's
  // rows are requested: with one table its phase test could not tell the two tiles apart.
  alignas(16) int32_t rowbuf[2][kTileTokens];
  uint32_t maskbuf[4][4];            // producer -> dequant: usable rows of each quarter, entry k % 4
  uint32_t stage_cnt[kPairStages];   // dequant warps done with a ring stage (2 per fill)
  uint32_t stage_req[kPairStages];   // fills requested per stage (the abort path waits for the last)
  uint32_t vmask[4][4];              // dequant -> softmax: usable rows of the tile, entry k % 4
  alignas(16) float red[4][32];      // softmax group: per-warp partial reductions
  int vote[8];
  int need_rescale;
};

template <int NH>
constexpr size_t pair_smem_bytes() {
  return 1024 + kPairVBytes + kPairQAtoms * NH * 128 + 2 * 128 * NH * 2 + 2 * 128 * NH * 4 + kPairRingBytes +
         sizeof(PairSmem);
}
static_assert(pair_smem_bytes<32>() <= 232448, "pair CTA exceeds the 227 KB shared-memory limit");
static_assert(kPairTmemS + 2 * 32 + 4 * 32 <= (int)kPairTmemCols, "TMEM columns");

// ---------------------------------------------------------------- partner exchange
// The partial scores go to the partner as asynchronous remote stores whose bytes complete on the
// partner's mbarrier (no fence: the receiver sees the data once the phase completes). The receiver
// tells the sender that a buffer has been read with a relaxed remote arrival, issued after every
// value read from it has been used.
__device__ __forceinline__ void st_async_u4(uint32_t remote_addr, const uint32_t* v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(remote_addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint64_t* bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(map_shared_rank(smem_u32(bar), rank))
               : "memory");
}

// Ring stage of quarter q of tile k: the ring holds two tiles, by tile parity.
__device__ __forceinline__ int pair_stage(int64_t k, int q) { return (int)(k & 1) * 4 + q; }

// Request the 32 rows of quarter q of tile k into its stage (8 gather4 copies, lanes 0..7) once the
// producers have resolved them. Returns false on timeout/abort.
__device__ __forceinline__ bool pair_issue_stage(const DecodeParams& p, PairSmem* sm, uint8_t* ring, int64_t k, int q,
                                                 int lane) {
  const int st = pair_stage(k, q);
  bool good = true;
  if (lane == 0) {
    good = wait(sm, &sm->rows_full[k & 1], (uint32_t)((k >> 1) & 1), p.status);
    if (good) {
      ++sm->stage_req[st];
      mbar_arrive_expect_tx(&sm->ring_full[st], (uint32_t)kPairStageBytes);
    }
  }
  good = __shfl_sync(0xffffffffu, good, 0);
  if (!good) return false;
  if (lane < 8) {
    const int4 r = *reinterpret_cast<const int4*>(&sm->rowbuf[k & 1][q * 32 + 4 * lane]);
    gather4(ring + st * kPairStageBytes + lane * 4 * kRowBytes, &p.cache_map, r.x, r.y, r.z, r.w, &sm->ring_full[st]);
  }
  __syncwarp();   // every lane has read its row numbers before the table is released
  if (lane == 0) mbar_arrive(&sm->rows_empty[k & 1]);
  return true;
}

// ---------------------------------------------------------------- dequant
// Warp (q, s): tile rows 32q..32q+31 (TMEM lane quarter q), the half's 64-dim groups 2s and 2s+1
// and rope dims 32 half + 16s .. + 15. Pass A converts the rows into K buffer k % 2 of TMEM; pass B
// copies the latent part of K into the V tile once PV of the previous tile is done with those rows.
// Pass A runs one tile ahead of pass B (A(k+1) before B(k)): K is double-buffered, so converting the
// next tile does not wait for the softmax and PV of the current one.
__device__ void pair_dequant(const DecodeParams& p, PairSmem* sm, uint8_t* ring, uint8_t* vtile, int64_t t_begin,
                             int64_t t_end, int warp, int half) {
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int s = (warp - 4) >> 2;
  const int row = 32 * q + lane;
  const uint32_t tmem_row = sm->tmem_base + ((uint32_t)(32 * q) << 16);
  const int64_t n = t_end - t_begin;
  // the sub-half 0 warps request the first two tiles' fills
  if (s == 0) {
    for (int64_t k0 = 0; k0 < 2 && k0 < n; ++k0)
      if (!pair_issue_stage(p, sm, ring, k0, q, lane)) return;
  }
  auto pass_a = [&](int64_t k) -> bool {
    const int st = pair_stage(k, q);
    bool good = true;
    if (lane == 0) {
      good = wait(sm, &sm->ring_full[st], (uint32_t)((k >> 1) & 1), p.status);
      // K buffer k % 2 may be rewritten once QK of tile k-2 is done (pass B(k-2) ran before this)
      if (good && k >= 2) good = wait(sm, &sm->qk_done[k & 1], (uint32_t)(((k - 2) >> 1) & 1), p.status);
    }
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) return false;
    __syncwarp();
    tc_fence_after();
    const uint8_t* rowp = ring + st * kPairStageBytes + lane * kRowBytes;
    const uint32_t kcol = (uint32_t)((k & 1) * kPairKCols);
    const uint32_t mask = sm->maskbuf[k & 3][q];
    // the 8 block scales of this warp's two groups: one 8-byte load
    const uint2 sc = *reinterpret_cast<const uint2*>(rowp + kScaleOff + 16 * half + 8 * s);
    uint32_t r[32];
#pragma unroll 1
    for (int gi = 0; gi < 2; ++gi) {
      const int l = 2 * s + gi;   // group within the half
      convert_group(rowp, 4 * half + l, gi == 0 ? sc.x : sc.y, r);
      __syncwarp();
      tmem_st32(tmem_row + kcol + 32 * l, r);
    }
    {
      // rope dims 32 half + 16 s .. + 15 (the half's 32 rope dims, 16 per sub-half): 16 E4M3 bytes
      // -> 8 fp16 pairs, K columns 128 + 8 s
      const uint4 v = *reinterpret_cast<const uint4*>(rowp + kRopeOff + 32 * half + 16 * s);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t rr[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rr[2 * i] = e4m3x2_to_f16x2(w[i] & 0xFFFFu);
        rr[2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
      }
      __syncwarp();
      tmem_st8(tmem_row + kcol + 128 + 8 * s, rr);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (s == 0) {
        sm->vmask[k & 3][q] = mask;
        mbar_arrive(&sm->mask_full[k & 3]);
      }
      mbar_arrive(&sm->kv_ready[k & 1]);
    }
    // refill: the second warp done with the stage requests tile k+2's rows into it
    uint32_t old = 0;
    if (lane == 0)
      asm volatile("atom.add.acq_rel.cta.shared::cta.u32 %0, [%1], 1;" : "=r"(old) : "r"(smem_u32(&sm->stage_cnt[st])) : "memory");
    old = __shfl_sync(0xffffffffu, old, 0);
    if ((old & 1u) && k + 2 < n && !pair_issue_stage(p, sm, ring, k + 2, q, lane)) return false;
    return true;
  };
  auto pass_b = [&](int64_t k) -> bool {
    bool good = true;
    if (lane == 0) good = wait(sm, &sm->vfree[q], (uint32_t)((k & 1) ^ 1), p.status);
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) return false;
    __syncwarp();
    tc_fence_after();
    const uint32_t kcol = (uint32_t)((k & 1) * kPairKCols);
    uint32_t r[32];
#pragma unroll 1
    for (int gi = 0; gi < 2; ++gi) {
      const int l = 2 * s + gi;
      tmem_ld32(tmem_row + kcol + 32 * l, r);
      tmem_wait_ld();
      uint8_t* vrow = vtile + l * 16384 + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(vrow + ((c ^ (row & 7)) << 4)) = make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->v_ready);
    return true;
  };
  if (n == 0 || !pass_a(0)) return;
  for (int64_t k = 0; k < n; ++k) {
    if (k + 1 < n && !pass_a(k + 1)) return;
    if (!pass_b(k)) return;
  }
}

// ---------------------------------------------------------------- MMA issue
// Two issuing threads per CTA (a single thread issuing every UMMA of a tile was the step that set
// the pace): warp 1 issues QK(k) = K half x q half into S buffer k % 2 (18 UMMAs of K = 16),
// warp 2 issues PV(k): for each of the half's two 128-dim M-blocks, the V
// rows times [P_hi | P_lo] (N = 2 NH) into [O_hi | O_lo], which the epilogue adds. One UMMA thus
// reads each V block once for both parts of P (the split kernel, with no TMEM left for a second
// O, reads it twice), halving the PV UMMAs and their shared-memory reads. When a tile starts a new
// unit its q image is requested once QK of the previous tile is done.
template <int NH>
__device__ void pair_qk_issuer(const DecodeParams& p, PairSmem* sm, uint8_t* qs, int64_t t_begin, int64_t t_end,
                               int half) {
  constexpr uint32_t kIdQK = idesc_f16(128, NH, false, false, false);
  constexpr uint32_t kAtom = (uint32_t)NH * 128u;
  const uint32_t tmem = sm->tmem_base;
  const uint64_t qd = sdesc(smem_u32(qs), 16, 1024, SW_128B);
  const int64_t n = t_end - t_begin;
  int64_t q_copies = 0;
  // this half's q atoms: latent atoms 4 half .. 4 half + 3, then the rope atom 8
  auto request_q = [&](int64_t unit) {
    const uint8_t* src = p.q16 + unit * (int64_t)(9u * kAtom);
    mbar_arrive_expect_tx(&sm->q_full, 5u * kAtom);
    bulk_g2s(qs, src + 4u * half * kAtom, 4u * kAtom, &sm->q_full);
    bulk_g2s(qs + 4u * kAtom, src + 8u * kAtom, kAtom, &sm->q_full);
    ++q_copies;
  };
  if (n > 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // q16 comes from the prep grid
  for (int64_t k = 0; k < n; ++k) {
    const TileInfo ti = tile_info(p, t_begin + k, t_begin, t_end);
    bool ok = true;
    if (ti.first) {
      // the q buffer is free once QK(k-1) has completed
      if (k > 0) ok = wait(sm, &sm->qk_done[(k - 1) & 1], (uint32_t)(((k - 1) >> 1) & 1), p.status);
      if (ok) {
        request_q(ti.unit);
        ok = wait(sm, &sm->q_full, (uint32_t)((q_copies - 1) & 1), p.status);
      }
    }
    if (ok) ok = wait(sm, &sm->kv_ready[k & 1], (uint32_t)((k >> 1) & 1), p.status);
    if (ok && k >= 2) ok = wait(sm, &sm->s_free[k & 1], (uint32_t)(((k - 2) >> 1) & 1), p.status);
    if (!ok) break;
    tc_fence_after();
    const uint32_t s_col = tmem + kPairTmemS + (uint32_t)(k & 1) * NH;
    const uint32_t kcol = tmem + (uint32_t)((k & 1) * kPairKCols);
    // latent dims 256 half .. + 255 (K-steps 16 half + x), then rope dims 32 half .. + 31 (K-steps
    // 32 + 2 half, 33 + 2 half): the split kernel's steps of this half, in its order
#pragma unroll
    for (int x = 0; x < 18; ++x) {
      const int ks = x < 16 ? 16 * half + x : 32 + 2 * half + (x - 16);   // K-step of the full contraction
      const int atom = x < 16 ? (x >> 2) : 4;                              // atom within this half's q image
      const uint64_t bq = qd + (uint64_t)(((uint32_t)atom * kAtom + (ks & 3) * 32) >> 4);
      umma_ts(s_col, kcol + 8 * x, bq, kIdQK, x > 0 ? 1u : 0u);
    }
    umma_commit(&sm->qk_done[k & 1]);
  }
  // never leave with a q copy in flight (abort path)
  if (q_copies > 0) mbar_wait(&sm->q_full, (uint32_t)((q_copies - 1) & 1), nullptr, kWaitTimeoutNs);
  umma_commit(&sm->drain);
  mbar_wait(&sm->drain, 0, nullptr, kWaitTimeoutNs);
}

template <int NH>
__device__ void pair_pv_issuer(const DecodeParams& p, PairSmem* sm, uint8_t* vtile, uint8_t* ps, int64_t t_begin,
                               int64_t t_end) {
  constexpr uint32_t kIdPV = idesc_f16(128, 2 * NH, true, true, false);
  constexpr uint32_t kPSw = (NH == 32) ? SW_128B : SW_64B;   // a token row of [P_hi | P_lo]: 2 NH fp16
  constexpr uint32_t kPSbo = (NH == 32) ? 1024 : 512;        // 8 token rows
  const uint32_t o_col = sm->tmem_base + kPairTmemS + 2 * NH;
  const uint64_t vd = sdesc(smem_u32(vtile), 16384, 1024, SW_128B);
  const uint64_t pd0 = sdesc(smem_u32(ps), 16384, kPSbo, kPSw);
  const int64_t n = t_end - t_begin;
  int64_t ofree_waits = 0;
  for (int64_t k = 0; k < n; ++k) {
    const TileInfo ti = tile_info(p, t_begin + k, t_begin, t_end);
    bool ok = wait(sm, &sm->p_full, (uint32_t)(k & 1), p.status);
    if (ok) ok = wait(sm, &sm->v_ready, (uint32_t)(k & 1), p.status);
    if (ok && ti.first && k > 0) ok = wait(sm, &sm->o_free, (uint32_t)(ofree_waits++ & 1), p.status);
    if (!ok) break;
    tc_fence_after();
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int ks = 2 * w + kk;
          const uint64_t a = vd + (uint64_t)((mi * 32768 + ks * 2048) >> 4);
          const uint64_t bdesc = pd0 + (uint64_t)((ks * 2 * kPSbo) >> 4);
          umma_ss(o_col + mi * 2 * NH, a, bdesc, kIdPV, (ti.first && ks == 0) ? 0u : 1u);
        }
      }
      umma_commit(&sm->vfree[w]);
    }
    if (ti.last) umma_commit(&sm->o_done);
  }
  umma_commit(&sm->drain);
  mbar_wait(&sm->drain, 0, nullptr, kWaitTimeoutNs);
}

// ---------------------------------------------------------------- softmax / epilogue
// Eight softmax warps: warp 12 + 4 hh + q takes tile rows 32q..32q+31 (TMEM lane quarter q) and
// heads hh NH/2 .. hh NH/2 + NH/2 - 1 (head half hh), so a thread follows one row through half the
// heads (one thread per row and all heads left the group latency-bound). Per tile: load this CTA's
// partial scores of the thread's heads from S buffer k % 2 and send them to the partner (row r of
// its xbuf), take the partner's from this CTA's xbuf, and add the two in the split kernel's order
// (half 0's + half 1's), so both CTAs hold the same scores and run the same softmax (same maxima,
// P and sums). Tile k+1's scores are sent as soon as P of tile k is out. Each CTA rescales and, at a
// segment's end, writes its own 256 dims of O; half 0 writes the (max, sum) partial.
constexpr int kPairSoftmaxThreads = 256;
__device__ __forceinline__ void pair_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool pair_sync_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
template <int HT>
__device__ __forceinline__ void tmem_ld_heads(uint32_t taddr, uint32_t (&r)[HT]) {
  if constexpr (HT == 16) tmem_ld16(taddr, r);
  else tmem_ld8(taddr, r);
}
template <int HT>
__device__ __forceinline__ void tmem_st_heads(uint32_t taddr, const uint32_t (&r)[HT]) {
  if constexpr (HT == 16) tmem_st16(taddr, r);
  else tmem_st8(taddr, r);
}

template <int NH>
__device__ bool pair_softmax(const DecodeParams& p, PairSmem* sm, uint8_t* ps, float* xbuf, int64_t t_begin,
                             int64_t t_end, int64_t pair, int half) {
  constexpr int HT = NH / 2;                            // heads per thread
  constexpr int kRowChunks = NH / 4;                    // 16-byte chunks of a score row
  constexpr int kTC = HT / 4;                           // of which this thread's
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, hh = (warp - 12) >> 2, w8 = warp - 12;
  const int row = 32 * q + lane, h0 = hh * HT;
  const uint32_t partner = (uint32_t)(half ^ 1);
  const uint32_t tmem_lane = sm->tmem_base + ((uint32_t)(32 * q) << 16);
  const uint32_t o_col = kPairTmemS + 2 * NH;
  const float kNegInf = __int_as_float(0xff800000);
  // row r of xbuf[b]: kRowChunks 16-byte chunks, chunk c stored at c ^ (r % kRowChunks)
  constexpr uint32_t kXBytes = 128u * NH * 4u;
  uint8_t* xrow = reinterpret_cast<uint8_t*>(xbuf) + row * NH * 4;
  const uint32_t xrow_remote = map_shared_rank(smem_u32(xrow), partner);
  const uint32_t xfull_remote = map_shared_rank(smem_u32(&sm->x_full[0]), partner);
  const int64_t n = t_end - t_begin;
  // Send this CTA's partial scores of tile k (row, the thread's heads) into the partner's
  // xbuf[k % 2] once QK(k) is done and the partner has read what was sent there for tile k-2, and
  // arm this CTA's receive of the partner's (x_full[k % 2]: its phase for tile k-2 is complete).
  auto send = [&](int64_t k) -> bool {
    const int xb = (int)(k & 1);
    if (threadIdx.x == 384) mbar_arrive_expect_tx(&sm->x_full[xb], kXBytes);
    bool good = true;
    if (lane == 0) {
      good = wait(sm, &sm->qk_done[k & 1], (uint32_t)((k >> 1) & 1), p.status);
      if (good && k >= 2) good = wait(sm, &sm->x_free[xb], (uint32_t)(((k - 2) >> 1) & 1), p.status);
    }
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) return false;
    __syncwarp();
    tc_fence_after();
    uint32_t own[HT];
    tmem_ld_heads<HT>(tmem_lane + kPairTmemS + (uint32_t)(k & 1) * NH + h0, own);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < kTC; ++c) {
      const int cc = hh * kTC + c;
      st_async_u4(xrow_remote + xb * kXBytes + ((cc ^ (row % kRowChunks)) << 4), own + 4 * c, xfull_remote + xb * 8u);
    }
    return true;
  };
  float l_part[HT];
  float qscale = 0.f;
  int64_t seg = 0;
  bool ok = true;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // qscale comes from the prep kernel
  if (n > 0 && pair_sync_any(!send(0))) ok = false;
  for (int64_t g = t_begin; g < t_end && ok; ++g) {
    const int64_t k = g - t_begin;
    const TileInfo ti = tile_info(p, g, t_begin, t_end);
    const int xb = (int)(k & 1);
    if (ti.first) {
      qscale = p.qscale[ti.unit];
#pragma unroll
      for (int j = 0; j < HT; ++j) l_part[j] = 0.f;
      if (threadIdx.x < 384 + 32) sm->m_used[threadIdx.x - 384] = kNegInf;
    }
    // row masks of tile k, and the partner's partial scores of tile k (QK(k) is done: sent)
    if (lane == 0 && wait(sm, &sm->mask_full[k & 3], (uint32_t)((k >> 2) & 1), p.status))
      wait(sm, &sm->x_full[xb], (uint32_t)((k >> 1) & 1), p.status);
    if (pair_sync_any(sm->abort != 0)) {
      ok = false;
      break;
    }
    tc_fence_after();
    __syncwarp();
    // ---- this CTA's partial scores (loaded again: they were sent, not kept)
    uint32_t own[HT];
    tmem_ld_heads<HT>(tmem_lane + kPairTmemS + (uint32_t)(k & 1) * NH + h0, own);
    tmem_wait_ld();
    // the row mask of tile k: entry k % 4 is rewritten by pass A of tile k+4, which waits for QK(k+2),
    // which waits for the release below
    const bool valid = (sm->vmask[k & 3][q] >> lane) & 1u;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->s_free[k & 1]);   // S buffer k % 2 read (8 warps): QK(k+2) may overwrite it
    float z[HT];
#pragma unroll
    for (int c = 0; c < kTC; ++c) {
      const int cc = hh * kTC + c;
      const uint4 v = *reinterpret_cast<const uint4*>(xrow + xb * kXBytes + ((cc ^ (row % kRowChunks)) << 4));
      const uint32_t other[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)   // half 0's partial + half 1's (fp32 addition is commutative)
        z[4 * c + i] = valid ? (__uint_as_float(own[4 * c + i]) + __uint_as_float(other[i])) * qscale : kNegInf;
    }
    // every value read from xbuf[xb] has been used: the partner may send tile k+2 into it
    __syncwarp();
    if (lane == 0) mbar_arrive_remote_relaxed(&sm->x_free[xb], partner);
    // ---- lazy running max (as in the split kernel), voted over the eight warps
    bool raise = ti.first;
    if (!raise) {
      bool exceed = false;
#pragma unroll
      for (int j = 0; j < HT; j += 4) {
        const float4 mv = *reinterpret_cast<const float4*>(&sm->m_used[h0 + j]);
        exceed |= (z[j] > mv.x + kLazy) | (z[j + 1] > mv.y + kLazy) | (z[j + 2] > mv.z + kLazy) | (z[j + 3] > mv.w + kLazy);
      }
      const int wv = __any_sync(0xffffffffu, exceed) ? 1 : 0;
      if (lane == 0) sm->vote[w8] = wv;
      pair_sync();
      int any = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) any |= sm->vote[i];
      raise = any != 0;
    }
    if (raise) {
#pragma unroll
      for (int j = 0; j < HT; j += 4) {
        float4 wm;
        wm.x = redux_max(z[j]);
        wm.y = redux_max(z[j + 1]);
        wm.z = redux_max(z[j + 2]);
        wm.w = redux_max(z[j + 3]);
        if (lane == 0) *reinterpret_cast<float4*>(&sm->red[q][h0 + j]) = wm;
      }
      pair_sync();
      if (w8 == 0) {
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
      pair_sync();
#pragma unroll
      for (int j = 0; j < HT; j += 4) {
        const float4 av = *reinterpret_cast<const float4*>(&sm->alpha[h0 + j]);
        l_part[j] *= av.x; l_part[j + 1] *= av.y; l_part[j + 2] *= av.z; l_part[j + 3] *= av.w;
      }
    }
    // ---- P(k) replaces P(k-1) once PV(k-1) has finished (its last commit covers all its UMMAs)
    if (k >= 1) {
      if (lane == 0) wait(sm, &sm->vfree[3], (uint32_t)((k - 1) & 1), p.status);
      __syncwarp();
      tc_fence_after();
    }
#pragma unroll
    for (int c = 0; c < HT / 8; ++c) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const int j = 8 * c + i;
        const float m0 = sm->m_used[h0 + j], m1 = sm->m_used[h0 + j + 1];
        const float p0 = (m0 == kNegInf) ? 0.f : ex2_approx(z[j] - m0);
        const float p1 = (m1 == kNegInf) ? 0.f : ex2_approx(z[j + 1] - m1);
        l_part[j] += p0;
        l_part[j + 1] += p1;
        const __half2 ph = __floats2half2_rn(p0, p1);
        const float2 fh = __half22float2(ph);
        const __half2 pl = __floats2half2_rn(p0 - fh.x, p1 - fh.y);
        hi[i >> 1] = *reinterpret_cast<const uint32_t*>(&ph);
        lo[i >> 1] = *reinterpret_cast<const uint32_t*>(&pl);
      }
      // row r of [P_hi | P_lo]: 16-byte chunk c holds P_hi of heads 8c..8c+7, chunk c + NH / 8 the
      // same heads' P_lo; 128-byte swizzle for NH = 32 (128-byte rows), 64-byte for NH = 16
      const int ch = h0 / 8 + c;
      const int off_hi = NH == 32 ? row * 128 + ((ch ^ (row & 7)) << 4) : row * 64 + ((ch ^ ((row >> 1) & 3)) << 4);
      const int off_lo = NH == 32 ? row * 128 + (((ch + 4) ^ (row & 7)) << 4) : row * 64 + (((ch + 2) ^ ((row >> 1) & 3)) << 4);
      *reinterpret_cast<uint4*>(ps + off_hi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(ps + off_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();
    // ---- a raised reference: O^T[dim, h] *= alpha[h] for the thread's heads, in both parts of this
    // half's two M-blocks, before PV(k)
    if (raise && sm->need_rescale && !ti.first) {
#pragma unroll 1
      for (int part = 0; part < 4; ++part) {
        const uint32_t col = o_col + (uint32_t)part * NH + h0;   // M-block part / 2, P_hi / P_lo part % 2
        uint32_t r[HT];
        tmem_ld_heads<HT>(tmem_lane + col, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < HT; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * sm->alpha[h0 + j]);
        tmem_st_heads<HT>(tmem_lane + col, r);
      }
      tmem_wait_st();
      tc_fence_before();
    }
    mbar_arrive(&sm->p_full);
    // ---- the next tile's exchange: after P(k), so PV(k) never waits for QK(k+1). A send that gives
    // up has set the abort flag, which the whole group reads at the next tile's barrier.
    if (k + 1 < n) (void)send(k + 1);

    if (ti.last) {
      // ---- epilogue: this half's dims of the segment's unnormalised partial
      if (lane == 0) wait(sm, &sm->o_done, (uint32_t)(seg & 1), p.status);
      if (pair_sync_any(sm->abort != 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t slot = pair + ti.unit;
      float* po = p.part_o + slot * (int64_t)NH * kLatent;
      {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = j < HT ? l_part[j] : 0.f;
        const float ws = warp_transpose_reduce<1>(v);   // lane j < HT: the warp's sum for head h0 + j
        if (lane < HT) sm->red[q][h0 + lane] = ws;
      }
      pair_sync();
      const int st = threadIdx.x - 384;
      if (half == 0 && st < NH) {
        const float lsum = sm->red[0][st] + sm->red[1][st] + sm->red[2][st] + sm->red[3][st];
        p.part_ml[(slot * NH + st) * 2 + 0] = sm->m_used[st];
        p.part_ml[(slot * NH + st) * 2 + 1] = lsum;
      }
      __syncwarp();
#pragma unroll 1
      for (int mb = 0; mb < 2; ++mb) {
        uint32_t rh[HT], rl[HT];   // O_hi, O_lo of M-block mb, the thread's heads
        tmem_ld_heads<HT>(tmem_lane + o_col + mb * 2 * NH + h0, rh);
        tmem_ld_heads<HT>(tmem_lane + o_col + mb * 2 * NH + NH + h0, rl);
        tmem_wait_ld();
        const int dim = 256 * half + mb * 128 + row;
#pragma unroll
        for (int j = 0; j < HT; ++j) po[(int64_t)(h0 + j) * kLatent + dim] = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
      }
      tc_fence_before();
      mbar_arrive(&sm->o_free);
      pair_sync();
      ++seg;
    }
  }
  return ok;
}

template <int NH>
__global__ void __launch_bounds__(kPairThreads, 1) decode_pair_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* vtile = base;                                   // 65536
  uint8_t* qs = vtile + kPairVBytes;                       // 5 atoms x NH x 128 B
  uint8_t* ps = qs + kPairQAtoms * NH * 128;               // P_hi, P_lo: 2 x 128 x NH x 2 B
  float* xbuf = reinterpret_cast<float*>(ps + 2 * 128 * NH * 2);   // the partner's partial scores: 2 x 128 x NH fp32
  uint8_t* ring = reinterpret_cast<uint8_t*>(xbuf) + 2 * 128 * NH * 4;
  PairSmem* sm = reinterpret_cast<PairSmem*>(ring + kPairRingBytes);

  const int warp = threadIdx.x >> 5;
  const int half = (int)cluster_ctarank();
  const int64_t pair = blockIdx.x >> 1;
  // Every decode CTA is resident once all of them reach this point, so letting the merge grid be
  // scheduled now cannot take resources a decode CTA still needs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t t_begin = range_begin(p, pair);
  const int64_t t_end = range_begin(p, pair + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPairStages; ++i) {
      mbar_init(&sm->ring_full[i], 1);
      sm->stage_cnt[i] = 0;
      sm->stage_req[i] = 0;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->rows_full[b], 2);
      mbar_init(&sm->rows_empty[b], 4);
      mbar_init(&sm->kv_ready[b], 8);
      mbar_init(&sm->qk_done[b], 1);
      mbar_init(&sm->s_free[b], 8);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&sm->mask_full[i], 4);
      mbar_init(&sm->vfree[i], 1);
    }
    mbar_init(&sm->v_ready, 8);
    mbar_init(&sm->p_full, kPairSoftmaxThreads);
    mbar_init(&sm->o_done, 1);
    mbar_init(&sm->o_free, kPairSoftmaxThreads);
    mbar_init(&sm->q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->x_full[b], 1);
      mbar_init(&sm->x_free[b], 8);
    }
    mbar_init(&sm->drain, 2);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm->tmem_base, kPairTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();   // both CTAs' barriers exist before either arrives on the other's

  if (warp == 0 || warp == 3) {
    producer_loop<false, 4, 2>(p, sm, t_begin, t_end, warp == 0 ? 0 : 1);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) pair_qk_issuer<NH>(p, sm, qs, t_begin, t_end, half);
    __syncwarp();
  } else if (warp == 2) {
    if ((threadIdx.x & 31) == 0) pair_pv_issuer<NH>(p, sm, vtile, ps, t_begin, t_end);
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    pair_dequant(p, sm, ring, vtile, t_begin, t_end, warp, half);
  } else if (warp >= 12) {   // 12..19
    pair_softmax<NH>(p, sm, ps, xbuf, t_begin, t_end, pair, half);
  }
  tc_fence_before();
  __syncthreads();
  // After an abort, never leave with gathers in flight: each stage has at most one fill outstanding
  // (a refill is requested only after the previous fill was consumed), the last one requested.
  if (threadIdx.x == 0 && sm->abort) {
    for (int i = 0; i < kPairStages; ++i)
      if (sm->stage_req[i] > 0) mbar_wait(&sm->ring_full[i], (sm->stage_req[i] - 1) & 1u, nullptr, kWaitTimeoutNs);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(sm->tmem_base, kPairTmemCols);
  }
  cluster_sync_all();   // neither CTA leaves while the other may still write into its shared memory
}

}  // namespace

static cudaError_t pair_attributes_once() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDevices && done[dev]) return cudaSuccess;
  err = cudaFuncSetAttribute(decode_pair_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pair_smem_bytes<32>());
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(decode_pair_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)pair_smem_bytes<16>());
  if (err == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev] = true;
  return err;
}

static cudaLaunchAttribute pair_cluster_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 2;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = 1;
  return a;
}

// Pairs of the decode grid that can be resident at once on the current device (0 on error).
int max_active_pairs(int heads_per_cta) {
  if (pair_attributes_once() != cudaSuccess) return 0;
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int cache[kMaxDevices][2] = {};   // value + 1; 0 = not computed yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int hi = heads_per_cta == 32 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDevices && cache[dev][hi] > 0) return cache[dev][hi] - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 64, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = hi ? pair_smem_bytes<32>() : pair_smem_bytes<16>();
  cudaLaunchAttribute attr[1] = {pair_cluster_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = hi ? cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel<32>, &cfg)
                           : cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel<16>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev][hi] = n + 1;
  return n;
}

// The pair grid alone (2 x p.ctas CTAs, clusters of 2), launched as a programmatic dependent of the
// q-prep grid; the caller launches the prep grid before and the merge grid after it.
cudaError_t launch_decode_pair(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t err = pair_attributes_once();
  if (err != cudaSuccess) return err;
  const bool h32 = p.heads_per_cta == 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * p.ctas), 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = h32 ? pair_smem_bytes<32>() : pair_smem_bytes<16>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0] = pair_cluster_attr();
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (h32) return cudaLaunchKernelEx(&cfg, decode_pair_kernel<32>, p);
  return cudaLaunchKernelEx(&cfg, decode_pair_kernel<16>, p);
}

}  // namespace nvfp4mla
