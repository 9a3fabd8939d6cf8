// Device helpers shared by the decode kernels (the split kernel in decode_kernel.cu and the pair
// kernel in decode_pair.cu): tile bookkeeping, bounded waits, index resolution and row gathers,
// the NVFP4 group conversion and warp reductions. Internal to the library; each including
// translation unit gets its own copy (anonymous namespace).
#pragma once
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4mla {
namespace {

using namespace ptx;

struct TileInfo {
  int64_t unit;     // virtual unit (query, head group)
  int local;        // tile index within the unit
  bool first, last; // first/last tile of this CTA's segment of the unit
};

// Tile numbers fit in 32 bits (the host rejects larger problems), so unsigned 32-bit division is used.
__device__ __forceinline__ TileInfo tile_info(const DecodeParams& p, int64_t g, int64_t t_begin, int64_t t_end) {
  TileInfo ti;
  const uint32_t u = (uint32_t)g / (uint32_t)p.tiles_per_unit;
  ti.unit = u;
  ti.local = (int)((uint32_t)g - u * (uint32_t)p.tiles_per_unit);
  ti.first = (g == t_begin) || (ti.local == 0);
  ti.last = (g == t_end - 1) || (ti.local == p.tiles_per_unit - 1);
  return ti;
}

template <class S>
__device__ __forceinline__ void fail(S* sm, int32_t* status) {
  if (!sm->abort) {
    sm->abort = 1;
    if (status != nullptr) atomicAdd(status + 2, 1);
  }
}

template <class S>
__device__ __forceinline__ bool wait(S* sm, uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait(bar, parity, &sm->abort, kWaitTimeoutNs)) return true;
  fail(sm, status);
  return false;
}

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Softmax-group barrier that also ORs a flag over the group, so every thread gets the same answer
// (the abort flag can be set by another warp at any time; reading it after a plain barrier could
// let one warp leave while the others wait at the next barrier).
__device__ __forceinline__ bool named_sync_softmax_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Stream-K ranges: the tiles of all units, cut into p.ctas contiguous ranges (CTAs, or pairs of
// CTAs), the first total_tiles % ctas of them one tile longer. The ranges launched last are the
// ones that can start late (on SMs the q-prep grid still holds), so they get the shorter shares.
__device__ __forceinline__ int64_t range_begin(const DecodeParams& p, int64_t r) {
  const int64_t base = p.total_tiles / p.ctas, extra = p.total_tiles % p.ctas;
  return r * base + (r < extra ? r : extra);
}
// The range that holds tile g.
__device__ __forceinline__ int64_t range_of_tile(const DecodeParams& p, int64_t g) {
  const int64_t base = p.total_tiles / p.ctas, extra = p.total_tiles % p.ctas;
  const int64_t split = extra * (base + 1);
  return g < split ? g / (base + 1) : extra + (g - split) / base;
}

// Unit decomposition: virtual unit -> (b, j, head group)
__device__ __forceinline__ void split_unit(const DecodeParams& p, int64_t unit, int& b, int& j, int& hg) {
  hg = (int)(unit % p.head_groups);
  const int64_t u = unit / p.head_groups;
  b = (int)(u / p.Q);
  j = (int)(u - (int64_t)b * p.Q);
}

// ------------------------------------------------------------------ producer
// Two producer warps; warp pw owns ring stages 2pw and 2pw+1 of every tile.
// Rows are gathered by TMA tile::gather4 (four arbitrary cache rows per
// instruction; lanes 0..7 each issue one per 32-row stage). Unusable entries
// get row -1, which the TMA unit fills with zeros without reading memory, so
// every stage always lands exactly 32 x 352 bytes.
// Index resolution is software-pipelined two tiles ahead: while tile g's rows
// are issued, the page-table words of tile g+1 and the index words of tile g+2
// are already in flight.
struct TileIdx {
  int idx[2];     // this lane's entries of the warp's two 32-row stages
  uint32_t mem[2];  // folded queries: the entries' query-token bits
  int L, causal;  // sequence length, causal limit of the query
  int b;
};

template <bool kFold>
__device__ __forceinline__ void load_tile_idx(const DecodeParams& p, int64_t g, int lane, int q0, TileIdx& t) {
  const int64_t unit = g / p.tiles_per_unit;
  const int local = (int)(g - unit * p.tiles_per_unit);
  int b, j, hg;
  split_unit(p, unit, b, j, hg);
  t.b = b;
  t.L = __ldg(p.seq_lens + b);
  t.causal = t.L - p.Q + j;
  const int32_t* row = p.idx + ((int64_t)b * p.Q + j) * p.topk;
#pragma unroll
  for (int qq = 0; qq < 2; ++qq) {
    const int e = local * kTileTokens + (q0 + qq) * 32 + lane;
    t.idx[qq] = e < p.topk ? __ldg(row + e) : -1;
    t.mem[qq] = (kFold && e < p.topk) ? (uint32_t)__ldg(p.fold_member + (int64_t)b * p.topk + e) : 0u;
  }
}

__device__ __forceinline__ void load_tile_pages(const DecodeParams& p, const TileIdx& t, int (&pg)[2]) {
  const int32_t* pt_row = p.page_table + (int64_t)t.b * p.max_pages;
#pragma unroll
  for (int qq = 0; qq < 2; ++qq) {
    const int idx = t.idx[qq];
    const bool in_range = idx >= 0 && idx < t.L && idx <= t.causal;
    pg[qq] = (in_range && (idx >> 6) < p.max_pages) ? __ldg(pt_row + (idx >> 6)) : -1;
  }
}

__device__ __forceinline__ void gather4(void* dst, const CUtensorMap* map, int r0, int r1, int r2, int r3,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// kRowBufs row tables: tile k is published in table k % kRowBufs once every stage of tile
// k - kRowBufs (the table's previous tile) has been requested; kMaskDepth mask entries, tile k in
// entry k % kMaskDepth.
template <bool kFold, int kMaskDepth, int kRowBufs, class S>
__device__ void producer_loop(const DecodeParams& p, S* sm, int64_t t_begin, int64_t t_end, int pw) {
  const int lane = threadIdx.x & 31;
  const int q0 = 2 * pw;
  TileIdx A0, A1, A2;
  int pg0[2], pg1[2];
  if (t_begin < t_end) load_tile_idx<kFold>(p, t_begin, lane, q0, A0);
  if (t_begin + 1 < t_end) load_tile_idx<kFold>(p, t_begin + 1, lane, q0, A1);
  if (t_begin < t_end) load_tile_pages(p, A0, pg0);
  for (int64_t g = t_begin; g < t_end && !sm->abort; ++g) {
    const int64_t k = g - t_begin;
    const int b = (int)(k % kMaskDepth);
    const TileInfo ti = tile_info(p, g, t_begin, t_end);
    if (g + 1 < t_end) load_tile_pages(p, A1, pg1);
    if (g + 2 < t_end) load_tile_idx<kFold>(p, g + 2, lane, q0, A2);
    const int hg = (int)(ti.unit % p.head_groups);
    // The row table is free once every stage of its previous tile has been requested; by then the
    // masks entry b held (tile k - kMaskDepth) have been read too.
    const int rb = (int)(k % kRowBufs);
    bool good = true;
    if (lane == 0 && k >= kRowBufs)
      good = wait(sm, &sm->rows_empty[rb], (uint32_t)(((k - kRowBufs) / kRowBufs) & 1), p.status);
    good = __shfl_sync(0xffffffffu, good, 0);
    if (!good) break;
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int q = q0 + qq;
      const int idx = A0.idx[qq];
      const int page = pg0[qq];
      const bool in_range = idx >= 0 && idx < A0.L && idx <= A0.causal;
      const bool ok = in_range && page >= 0 && page < p.num_pages;
      if (hg == 0 && p.status != nullptr) {
        const int e = ti.local * kTileTokens + q * 32 + lane;
        const uint32_t nbi = __popc(__ballot_sync(0xffffffffu, idx != -1 && !in_range && e < p.topk));
        const uint32_t nbp = __popc(__ballot_sync(0xffffffffu, in_range && !ok));
        if (lane == 0 && nbi) atomicAdd(p.status + 0, (int)nbi);
        if (lane == 0 && nbp) atomicAdd(p.status + 1, (int)nbp);
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, ok);
      sm->rowbuf[rb][q * 32 + lane] = ok ? page * kPageTokens + (idx & 63) : -1;
      if (lane == 0) sm->maskbuf[b][q] = mask;
      if constexpr (kFold) {
        // query token jj of the fold may use the entry if it is listed for jj and within jj's causal range
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const bool use = ok && jj < p.fold_q && ((A0.mem[qq] >> jj) & 1u) && idx <= A0.L - p.fold_q + jj;
          const uint32_t mj = __ballot_sync(0xffffffffu, use);
          if (lane == 0) sm->maskq[b][q][jj] = mj;
        }
      }
    }
    __syncwarp();
    // (testing aid: withholding tile 1's table makes the waits on it expire)
    if (lane == 0 && !(p.withhold && k == 1)) mbar_arrive(&sm->rows_full[rb]);
    A0 = A1;
    A1 = A2;
    pg0[0] = pg1[0];
    pg0[1] = pg1[1];
  }
}

// ------------------------------------------------------------------ dequant
// One group = 64 values (32 nibble bytes) sharing four block scales (sw). Ring rows are 352 B
// apart, so the 16-byte loads see two-way bank conflicts; undoing a lane-dependent load order
// would cost more ALU work than the conflicts cost (the pass is bound by its conversions).
__device__ __forceinline__ void convert_group(const uint8_t* rowp, int g, uint32_t sw, uint32_t (&r)[32]) {
  const uint4 n0 = *reinterpret_cast<const uint4*>(rowp + 32 * g);
  const uint4 n1 = *reinterpret_cast<const uint4*>(rowp + 32 * g + 16);
  const uint32_t w[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
  for (int bb = 0; bb < 4; ++bb) {
    const uint32_t s2 = e4m3x2_to_f16x2(__byte_perm(sw, 0, bb * 0x11));   // (scale, scale)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t c[4];
      e2m1x8_to_f16x2x4(w[2 * bb + h], c);
#pragma unroll
      for (int i = 0; i < 4; ++i) r[8 * bb + 4 * h + i] = hmul2(c[i], s2);
    }
  }
}

// ------------------------------------------------------------------ softmax
// Maximum of v over the 32 lanes of the warp (every lane gets it).
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Transpose-reduce 32 values across a warp: afterwards lane l holds the reduction
// (over the 32 lanes) of element l. op: 0 = max, 1 = sum.
template <int OP>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      // keep half [i] (lower) or [i+s] (upper); send the other half
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = OP == 0 ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// Softmax group: thread t owns tile row t (a token) and all heads. The reference m of each head
// (the "running max") is kept lazily: it is raised only when a score exceeds it by more than
// kLazy = 15 (log2 units), so most tiles need one group vote instead of a max reduction, and
// P = 2^(z - m) stays <= 2^15, inside the fp16 range. When raised it is set to the tile's maximum
// (no headroom), so P keeps fp16's whole range below it: weights down to 2^-24 of the maximum's
// are represented, and the mass lost below that is at most topk * 2^-25 of the total. (A reference
// set above the maximum would cut the raises but move the underflow threshold up with it: with 8
// units of headroom, 2,047 tokens 17 units below a dominant one lost 1.5 % of the mass.)
constexpr float kLazy = 15.f;

}  // namespace
}  // namespace nvfp4mla
