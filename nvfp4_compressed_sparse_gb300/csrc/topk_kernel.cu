// indexer_topk kernel: the top-k positions of each query token's indexer logits, the index lists
// sparse_mla_decode reads.
//
// What is selected ("Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", section
// "Decode: TP4, and the copies it keeps": the indexer picks the top-2,048 positions of a query;
// "Prime Inference", translated page, "Native NVFP4 sparse MLA decode kernel": unused entries
// are -1): from the causal range 0..seq_len-Q+j of query j, the K largest logits, ties to the
// smaller position, NaN below every number; the list holds the positions in increasing order,
// -1 padded when the range is shorter than K.
//
// GB300 design: one 1024-thread CTA per query row; an exact radix select on order-preserving
// 32-bit keys, in three tiers that each verify their own precondition and hand the row to the
// next one when it fails:
//   1. sampled bound (rows up to 262,144 positions, K <= 4,096): a 12-bit histogram of a 1/16
//      sample (8 positions in every 128) gives a key bound with about 1.5 K keys of the row
//      expected above it; one sweep keeps every key at or above it (a single float compare per
//      logit) as a candidate in shared memory; with at least K and at most 8,192 candidates the
//      select finishes there (below);
//   2. full histogram (rows up to 262,144 positions): a 4,096-bin histogram of the keys' top 12
//      bits over the row gives the bin of the K-th largest key; a second sweep marks the
//      positions above that bin in a bitmap and keeps the bin's keys as candidates;
//   3. general: the remaining digits by sweeps over the row, then a position-ordered compaction
//      with one block scan of packed (greater, tie) counts per 8,192 positions.
// Finishing from candidates: the remaining digits of the threshold key T and the number R of
// keys equal to T that are taken come from histogram rounds over the candidates; candidates above
// T and equal to T go into two position bitmaps, and one block-wide scan over the bitmap words
// writes the positions in increasing order (the ties: the first R). The sweeps are coalesced
// 16-byte loads, 128 bytes per thread in flight.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4mla {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkPer = 8;                        // consecutive positions per thread per group
constexpr int kTkGroup = kTkThreads * kTkPer;    // positions per group (8,192)
constexpr int kTkCandCap = 8192;                 // candidates kept in shared memory (fast path)
constexpr int kTkMapWords = 8192;                // bitmap words: rows up to 262,144 positions (fast path)

// Unsigned order of the key = selection order of the float (NaN lowest, -0.0 below +0.0).
// The sign flip maps negative NaNs to [0, 0x007FFFFE] and positive NaNs to (0xFF800000, 2^32);
// one unsigned range test on k - key(-inf) sends both to 0.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  const uint32_t k = bits ^ ((uint32_t)((int32_t)bits >> 31) | 0x80000000u);
  return (k - 0x007FFFFFu) > 0xFF000001u ? 0u : k;
}

__device__ __forceinline__ void keys8(uint4 a, uint4 b, uint32_t (&k)[kTkPer]) {
  k[0] = order_key(a.x); k[1] = order_key(a.y); k[2] = order_key(a.z); k[3] = order_key(a.w);
  k[4] = order_key(b.x); k[5] = order_key(b.y); k[6] = order_key(b.z); k[7] = order_key(b.w);
}

// Keys of positions p0..p0+7 of the row; positions >= n get key 0 and valid = 0. kLastUse loads
// evict-first (the row's last sweep); otherwise the lines stay in L2 for the next sweep.
template <bool kLastUse = true>
__device__ __forceinline__ uint32_t load_keys(const float* row, int64_t p0, int64_t n, uint32_t (&k)[kTkPer]) {
  if (p0 + kTkPer <= n) {
    const uint4* p = reinterpret_cast<const uint4*>(row + p0);
    if (kLastUse) keys8(__ldcs(p), __ldcs(p + 1), k);
    else keys8(__ldg(p), __ldg(p + 1), k);
    return 0xFFu;
  }
  uint32_t valid = 0;
#pragma unroll
  for (int i = 0; i < kTkPer; ++i) {
    const bool in = p0 + i < n;
    k[i] = in ? order_key(__float_as_uint(kLastUse ? __ldcs(row + p0 + i) : __ldg(row + p0 + i))) : 0u;
    valid |= (in ? 1u : 0u) << i;
  }
  return valid;
}

// Block-wide exclusive prefix sum of v (1024 threads); *total gets the sum of all.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, s);
    if (lane >= s) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sums[lane];
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, s);
      if (lane >= s) w += y;
    }
    warp_sums[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
  *total = warp_sums[31];
  __syncthreads();         // warp_sums may be reused by the next scan
  return before;
}

struct TopkShared {
  alignas(16) uint32_t hist[4096];
  alignas(16) uint32_t mhist[4096];            // cluster: the first tier's sample histogram summed over the CTAs
  uint32_t m_local;                // cluster: this CTA's sample size
  uint32_t warp_sums[32];
  uint32_t found_digit, found_rem, cand_count;
  uint32_t cand_key[kTkCandCap];
  int32_t cand_pos[kTkCandCap];
  uint32_t gt_map_[kTkMapWords];   // positions whose key is above the threshold key
  uint32_t eq_map_[kTkMapWords];   // positions whose key equals it
};

__device__ __forceinline__ uint32_t* gt_map(TopkShared& sh) { return sh.gt_map_; }
__device__ __forceinline__ uint32_t* eq_map(TopkShared& sh) { return sh.eq_map_; }

// The digit of the rem-th largest key from a filled histogram (bins scanned from the top):
// updates prefix/pmask with the digit at `shift` and rem with the rank left inside its bin.
__device__ __forceinline__ void take_digit(TopkShared& sh, const uint32_t* hist, int bins, int shift,
                                           uint32_t& prefix, uint32_t& pmask, uint32_t& rem) {
  const int t = threadIdx.x;
  const int per = bins / kTkThreads > 0 ? bins / kTkThreads : 1;
  const int hi = bins - per * t;          // this thread owns bins [hi - per, hi)
  uint32_t mine = 0;
  if (hi > 0)
    for (int i = 1; i <= per; ++i) mine += hist[hi - i];
  uint32_t total;
  const uint32_t above = block_exclusive_scan(mine, sh.warp_sums, &total);   // counts in higher bins
  if (hi > 0 && above < rem && above + mine >= rem) {
    uint32_t cum = above;
    for (int i = 1; i <= per; ++i) {
      const uint32_t h = hist[hi - i];
      if (cum + h >= rem) {
        sh.found_digit = (uint32_t)(hi - i);
        sh.found_rem = rem - cum;
        break;
      }
      cum += h;
    }
  }
  __syncthreads();
  prefix |= sh.found_digit << shift;
  pmask |= (uint32_t)(bins - 1) << shift;
  rem = sh.found_rem;
  __syncthreads();
}

// Histogram of the digit at `shift` over the row's keys that match prefix under pmask.
template <bool kFiltered>
__device__ __forceinline__ void global_histogram(TopkShared& sh, const float* row, int64_t n, int shift, int bins,
                                                 uint32_t prefix, uint32_t pmask) {
  const int t = threadIdx.x;
  for (int i = t; i < bins; i += kTkThreads) sh.hist[i] = 0;
  __syncthreads();
  const uint32_t dmask = (uint32_t)(bins - 1);
  int64_t base = 0;
  // full sweeps of 4 groups: no per-position checks
#pragma unroll 1
  for (; base + 4 * kTkGroup <= n; base += 4 * kTkGroup) {
    uint4 a[4], b[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4* p = reinterpret_cast<const uint4*>(row + base + g * kTkGroup + t * kTkPer);
      a[g] = __ldg(p);
      b[g] = __ldg(p + 1);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t k[kTkPer];
      keys8(a[g], b[g], k);
#pragma unroll
      for (int i = 0; i < kTkPer; ++i)
        if (!kFiltered || (k[i] & pmask) == prefix) atomicAdd(&sh.hist[(k[i] >> shift) & dmask], 1u);
    }
  }
#pragma unroll 1
  for (; base < n; base += kTkGroup) {
    uint32_t k[kTkPer];
    const uint32_t v = load_keys(row, base + (int64_t)t * kTkPer, n, k);
#pragma unroll
    for (int i = 0; i < kTkPer; ++i)
      if (((v >> i) & 1u) && (!kFiltered || (k[i] & pmask) == prefix))
        atomicAdd(&sh.hist[(k[i] >> shift) & dmask], 1u);
  }
  __syncthreads();
}

// Appends the keys flagged in `bits` (key i at position p0 + i) to the candidate store with one
// shared atomic per warp: a warp scan of the per-lane counts gives every lane its slots. Called by
// all 32 lanes; slots past the store's capacity are counted but not written.
__device__ __forceinline__ void append_candidates(TopkShared& sh, uint32_t bits, const uint32_t (&keys)[kTkPer],
                                                  int32_t p0) {
  const int lane = threadIdx.x & 31;
  const uint32_t cnt = __popc(bits);
  uint32_t incl = cnt;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, s);
    if (lane >= s) incl += y;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  if (total == 0u) return;
  uint32_t base = 0;
  if (lane == 31) base = atomicAdd(&sh.cand_count, total);
  uint32_t slot = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
#pragma unroll
  for (int i = 0; i < kTkPer; ++i) {
    if ((bits >> i) & 1u) {
      if (slot < (uint32_t)kTkCandCap) {
        sh.cand_key[slot] = keys[i];
        sh.cand_pos[slot] = p0 + i;
      }
      ++slot;
    }
  }
}

// One element of the candidate sweep: above the top digit -> marked selected; returns whether it
// is a candidate (in the top digit's bin).
__device__ __forceinline__ bool classify(TopkShared& sh, uint32_t k, int32_t pos, uint32_t d1) {
  const uint32_t d = k >> 20;
  if (d > d1) atomicOr(&gt_map(sh)[pos >> 5], 1u << (pos & 31));
  return d == d1;
}

// Candidate sweep over positions [0, n) (row relative). With kFloatTest the hot loop tests each
// logit against f_lo, the smallest float whose key reaches the top digit d1 (valid for
// 8 <= d1 <= 0xFF8, where f_lo is a number and no NaN passes); the exact key is formed only for the few that pass.
// Float order equals key order except that -0.0 == +0.0 there, so the test passes a superset
// and classify() decides exactly.
template <bool kFloatTest>
__device__ __forceinline__ void candidate_sweep(TopkShared& sh, const float* row, int64_t n, uint32_t d1,
                                                float f_lo) {
  const int t = threadIdx.x;
  int64_t base = 0;
#pragma unroll 1
  for (; base + 4 * kTkGroup <= n; base += 4 * kTkGroup) {
    float4 a[4], c[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float4* p = reinterpret_cast<const float4*>(row + base + g * kTkGroup + t * kTkPer);
      a[g] = __ldcs(p);
      c[g] = __ldcs(p + 1);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float v[kTkPer] = {a[g].x, a[g].y, a[g].z, a[g].w, c[g].x, c[g].y, c[g].z, c[g].w};
      const int32_t p0 = (int32_t)(base + g * kTkGroup + t * kTkPer);
      uint32_t keys[kTkPer], bits = 0;
#pragma unroll
      for (int i = 0; i < kTkPer; ++i) {
        keys[i] = 0u;
        if (!kFloatTest || v[i] >= f_lo) {
          keys[i] = order_key(__float_as_uint(v[i]));
          if (classify(sh, keys[i], p0 + i, d1)) bits |= 1u << i;
        }
      }
      append_candidates(sh, bits, keys, p0);
    }
  }
#pragma unroll 1
  for (; base < n; base += kTkGroup) {
    uint32_t k[kTkPer], bits = 0;
    const int64_t p0 = base + (int64_t)t * kTkPer;
    const uint32_t v = load_keys(row, p0, n, k);
#pragma unroll
    for (int i = 0; i < kTkPer; ++i)
      if (((v >> i) & 1u) && classify(sh, k[i], (int32_t)(p0 + i), d1)) bits |= 1u << i;
    append_candidates(sh, bits, k, (int32_t)p0);
  }
}

// Histogram add for a warp whose lanes may hit the same bin (candidate keys crowd into a few
// bins): lanes with equal bins are grouped and one of them adds the group's count. Called by all
// 32 lanes.
__device__ __forceinline__ void hist_add_grouped(uint32_t* hist, uint32_t bin, bool active) {
  const uint32_t act = __ballot_sync(0xffffffffu, active);
  if (active) {
    const uint32_t peers = __match_any_sync(act, bin);
    if ((int)(__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
  }
}

// The rest of the select over the c candidates in shared memory, which hold every key of the
// row that can still be selected: the digits from d_start on (0: bits 31..20, 1: 19..8, 2: 7..0)
// of the threshold key T and the count R of ties taken, then the bitmaps and the list.
// clear_maps: start from empty bitmaps (else gt_map already holds the keys above the candidates).
__device__ void finish_from_candidates(TopkShared& sh, uint32_t c, int d_start, uint32_t prefix, uint32_t pmask,
                                       uint32_t rem, int W, bool clear_maps, int32_t* o) {
  const int t = threadIdx.x;
#pragma unroll 1
  for (int d = d_start; d < 3; ++d) {
    const int shift = d == 0 ? 20 : (d == 1 ? 8 : 0), bins = d < 2 ? 4096 : 256;
    for (int i = t; i < bins; i += kTkThreads) sh.hist[i] = 0;
    __syncthreads();
    for (uint32_t base = (uint32_t)(t & ~31); base < c; base += kTkThreads) {   // warp-uniform trip count
      const uint32_t i = base + (uint32_t)(t & 31);
      const uint32_t k = i < c ? sh.cand_key[i] : 0u;
      hist_add_grouped(sh.hist, (k >> shift) & (uint32_t)(bins - 1), i < c && (k & pmask) == prefix);
    }
    __syncthreads();
    take_digit(sh, sh.hist, bins, shift, prefix, pmask, rem);
  }
  const uint32_t T = prefix, R = rem;
  if (clear_maps) {
    for (int i = t; i < W; i += kTkThreads) gt_map(sh)[i] = 0, eq_map(sh)[i] = 0;
    __syncthreads();
  }
  for (uint32_t i = t; i < c; i += kTkThreads) {
    const uint32_t k = sh.cand_key[i];
    const int32_t pos = sh.cand_pos[i];
    if (k > T) atomicOr(&gt_map(sh)[pos >> 5], 1u << (pos & 31));
    else if (k == T) atomicOr(&eq_map(sh)[pos >> 5], 1u << (pos & 31));
  }
  __syncthreads();
  // emit in position order: a word's first slot = (selected bits before it) + min(tie bits
  // before it, R); its ties are taken while the tie rank stays below R
  const int wpt = (W + kTkThreads - 1) / kTkThreads;
  const int w0 = t * wpt, w1 = min(W, w0 + wpt);
  uint32_t g = 0, e = 0;
  for (int w = w0; w < w1; ++w) g += __popc(gt_map(sh)[w]), e += __popc(eq_map(sh)[w]);
  uint32_t tot;
  const uint32_t ex = block_exclusive_scan(g | (e << 16), sh.warp_sums, &tot);
  uint32_t gb = ex & 0xFFFFu, eb = ex >> 16;
  for (int w = w0; w < w1; ++w) {
    uint32_t gm = gt_map(sh)[w], em = eq_map(sh)[w];
    uint32_t slot = gb + (eb < R ? eb : R);
    gb += __popc(gm);
    uint32_t keep = eb < R ? R - eb : 0u, taken = 0;   // the lowest (R - eb) tie bits of this word
    eb += __popc(em);
    while (em != 0u && keep != 0u) {
      const uint32_t low = em & (0u - em);
      taken |= low;
      em ^= low;
      --keep;
    }
    uint32_t sel = gm | taken;
    while (sel != 0u) {
      const int bit = __ffs(sel) - 1;
      o[slot++] = w * 32 + bit;
      sel &= sel - 1u;
    }
  }
}

// First tier: a sample of the row (8 positions in every 128) bounds the K-th largest key from
// below, one sweep keeps every key at or above the bound as a candidate, and the select finishes
// in shared memory. The bound is chosen so that about 1.5 K keys of the row are expected above
// it; it is checked exactly (at least K candidates, at most the store's capacity), and on a miss
// the caller takes the next tier. Returns true when the list is written (block-uniform).
//
// kCluster: the C CTAs of a thread-block cluster share the row; CTA r samples and sweeps the r-th
// slice (a multiple of 8 positions). The sample histograms and sizes are summed through distributed
// shared memory (every CTA computes the same bound from the sum), each CTA keeps its slice's
// candidates, and the CTAs then append theirs to CTA 0's store, which finishes the select. Every
// decision is taken on cluster-wide values, so all CTAs return the same value; on a miss CTA 0
// alone takes the next tiers.
template <bool kCluster>
__device__ bool sample_select(TopkShared& sh, const float* row, int64_t n, int K, int32_t* o, uint32_t rank,
                              uint32_t csize) {
  namespace px = nvfp4mla::ptx;
  const int t = threadIdx.x;
  int64_t lo_r = 0, hi_r = n;
  if constexpr (kCluster) {
    const int64_t per = ((n + csize - 1) / csize + 7) & ~(int64_t)7;
    lo_r = min(n, (int64_t)rank * per);
    hi_r = min(n, lo_r + per);
  }
  for (int i = t; i < 4096; i += kTkThreads) sh.hist[i] = 0;
  if (t == 0) sh.cand_count = 0;
  __syncthreads();
  uint32_t mine = 0;
  for (int64_t p0 = lo_r + (int64_t)t * 128; p0 < hi_r; p0 += (int64_t)kTkThreads * 128) {
    uint32_t k[kTkPer];
    const uint32_t v = load_keys<false>(row, p0, hi_r, k);
#pragma unroll
    for (int i = 0; i < kTkPer; ++i)
      if ((v >> i) & 1u) atomicAdd(&sh.hist[k[i] >> 20], 1u);
    mine += __popc(v);
  }
  __syncthreads();
  uint32_t m;
  block_exclusive_scan(mine, sh.warp_sums, &m);
  const uint32_t* hist = sh.hist;
  if constexpr (kCluster) {
    if (t == 0) sh.m_local = m;
    px::cluster_sync_all();                        // every CTA's sample histogram and size are final
    // thread t sums bins 4t..4t+3 of every CTA (one 16-byte load per CTA, all issued before use)
    static_assert(4096 == 4 * kTkThreads, "one group of four bins per thread");
    const uint32_t hbase = px::smem_u32(sh.hist) + 16 * t, mbase = px::smem_u32(&sh.m_local);
    uint4 part[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      part[r] = r < (int)csize ? px::ld_dsmem_u4(px::map_shared_rank(hbase, r)) : make_uint4(0u, 0u, 0u, 0u);
    uint4 sum = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int r = 0; r < 8; ++r) sum.x += part[r].x, sum.y += part[r].y, sum.z += part[r].z, sum.w += part[r].w;
    *reinterpret_cast<uint4*>(&sh.mhist[4 * t]) = sum;
    m = 0;
    for (uint32_t r = 0; r < csize; ++r) m += px::ld_dsmem_u32(px::map_shared_rank(mbase, r));
    __syncthreads();
    hist = sh.mhist;
  }
  // rank (from the top) in the sample of the bound: ceil(1.5 K m / n) + 32
  const int64_t want = (3 * (int64_t)K * m + 2 * n - 1) / (2 * n) + 32;
  uint32_t db = 0;
  if (want <= (int64_t)m) {
    uint32_t prefix = 0, pmask = 0, rem = (uint32_t)want;
    take_digit(sh, hist, 4096, 20, prefix, pmask, rem);
    db = prefix >> 20;
  }
  if constexpr (kCluster) px::cluster_sync_all();   // no CTA reads another's histogram after this
  if (db < 8 || db > 0xFF8) return false;   // no usable bound (it would not be a number)
  const uint32_t lo = db << 20;
  const float f_lo = __uint_as_float(lo >= 0x80000000u ? (lo & 0x7FFFFFFFu) : ~lo);

  // the sweep: every key >= lo becomes a candidate (f_lo passes a superset, see candidate_sweep)
  int64_t base = lo_r;
#pragma unroll 1
  for (; base + 4 * kTkGroup <= hi_r; base += 4 * kTkGroup) {
    float4 a[4], c[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float4* p = reinterpret_cast<const float4*>(row + base + g * kTkGroup + t * kTkPer);
      a[g] = __ldcs(p);
      c[g] = __ldcs(p + 1);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float v[kTkPer] = {a[g].x, a[g].y, a[g].z, a[g].w, c[g].x, c[g].y, c[g].z, c[g].w};
      const int32_t p0 = (int32_t)(base + g * kTkGroup + t * kTkPer);
      uint32_t keys[kTkPer], bits = 0;
#pragma unroll
      for (int i = 0; i < kTkPer; ++i) {
        keys[i] = 0u;
        if (v[i] >= f_lo) {
          keys[i] = order_key(__float_as_uint(v[i]));
          if (keys[i] >= lo) bits |= 1u << i;
        }
      }
      append_candidates(sh, bits, keys, p0);
    }
  }
#pragma unroll 1
  for (; base < hi_r; base += kTkGroup) {
    uint32_t k[kTkPer], bits = 0;
    const int64_t p0 = base + (int64_t)t * kTkPer;
    const uint32_t v = load_keys(row, p0, hi_r, k);
#pragma unroll
    for (int i = 0; i < kTkPer; ++i)
      if (((v >> i) & 1u) && k[i] >= lo) bits |= 1u << i;
    append_candidates(sh, bits, k, (int32_t)p0);
  }
  __syncthreads();
  uint32_t c = sh.cand_count;
  if constexpr (kCluster) {
    // cluster-wide count and this CTA's offset in CTA 0's store
    px::cluster_sync_all();                        // every CTA's count is final
    const uint32_t cbase = px::smem_u32(&sh.cand_count);
    uint32_t total = 0, off = 0;
    bool over = false;
    for (uint32_t r = 0; r < csize; ++r) {
      const uint32_t cr = px::ld_dsmem_u32(px::map_shared_rank(cbase, r));
      over |= cr > (uint32_t)kTkCandCap;
      if (r < rank) off += cr;
      total += cr;
    }
    px::cluster_sync_all();                        // every count has been read
    if (over || total < (uint32_t)K || total > (uint32_t)kTkCandCap) return false;
    if (rank != 0) {
      const uint32_t kb = px::map_shared_rank(px::smem_u32(sh.cand_key), 0);
      const uint32_t pb = px::map_shared_rank(px::smem_u32(sh.cand_pos), 0);
      for (uint32_t i = t; i < c; i += kTkThreads) {
        px::st_dsmem_u32(kb + 4 * (off + i), sh.cand_key[i]);
        px::st_dsmem_u32(pb + 4 * (off + i), (uint32_t)sh.cand_pos[i]);
      }
    }
    px::cluster_sync_all();                        // CTA 0 holds every candidate
    if (rank != 0) return true;
    c = total;
  }
  if (c < (uint32_t)K || c > (uint32_t)kTkCandCap) return false;
  finish_from_candidates(sh, c, 0, 0u, 0u, (uint32_t)K, (int)((n + 31) >> 5), true, o);
  return true;
}

// kCluster: launched with clusters of C CTAs, cluster c selecting row c (see sample_select); the
// tiers after the first run in CTA 0 of the cluster alone.
template <bool kCluster>
__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(const float* __restrict__ logits, int64_t stride,
                                                             const int32_t* __restrict__ seq_lens, int Q, int K,
                                                             int32_t* __restrict__ out, int csize) {
  extern __shared__ __align__(16) unsigned char topk_smem[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(topk_smem);
  const uint32_t rank = kCluster ? nvfp4mla::ptx::cluster_ctarank() : 0u;
  const int64_t rowi = kCluster ? (int64_t)blockIdx.x / csize : (int64_t)blockIdx.x;
  const int b = (int)(rowi / Q), j = (int)(rowi - (int64_t)b * Q);
  int64_t n = (int64_t)__ldg(seq_lens + b) - Q + j + 1;
  if (n < 0) n = 0;
  if (n > stride) n = stride;
  int32_t* o = out + rowi * K;
  const int t = threadIdx.x;
  if (n <= K) {   // the whole range is selected
    if (rank == 0)
      for (int i = t; i < K; i += kTkThreads) o[i] = i < n ? i : -1;
    return;
  }
  const float* row = logits + rowi * stride;

  const bool maps_fit = n <= 32 * (int64_t)kTkMapWords;
  if (maps_fit && 2 * K <= kTkCandCap && sample_select<kCluster>(sh, row, n, K, o, rank, (uint32_t)csize)) return;
  if (rank != 0) return;
  __syncthreads();

  // ---- second tier: the top 12 bits of the K-th largest key, over the whole row
  uint32_t prefix = 0, pmask = 0;
  uint32_t rem = (uint32_t)K;   // rank (from the top) of the wanted key among those matching prefix
  global_histogram<false>(sh, row, n, 20, 4096, 0u, 0u);
  take_digit(sh, sh.hist, 4096, 20, prefix, pmask, rem);

  if (maps_fit) {
    // one more sweep marks the keys above that digit in a position bitmap and
    // keeps the keys in its bin as candidates; the rest of the select runs in shared memory.
    const int W = (int)((n + 31) >> 5);
    for (int i = t; i < W; i += kTkThreads) gt_map(sh)[i] = 0, eq_map(sh)[i] = 0;
    if (t == 0) sh.cand_count = 0;
    __syncthreads();
    const uint32_t d1 = prefix >> 20;
    if (d1 >= 8 && d1 <= 0xFF8) {   // f_lo finite or +inf; the digits between hold only NaN keys
      const uint32_t lo = d1 << 20;
      candidate_sweep<true>(sh, row, n, d1, __uint_as_float(lo >= 0x80000000u ? (lo & 0x7FFFFFFFu) : ~lo));
    } else {
      candidate_sweep<false>(sh, row, n, d1, 0.f);
    }
    __syncthreads();
    const uint32_t c = sh.cand_count;
    if (c <= (uint32_t)kTkCandCap) {
      finish_from_candidates(sh, c, 1, prefix, pmask, rem, W, false, o);
      return;
    }
  }

  // ---- general path: the remaining digits over the row in global memory
#pragma unroll 1
  for (int d = 1; d < 3; ++d) {
    const int shift = d == 1 ? 8 : 0, bins = d == 1 ? 4096 : 256;
    global_histogram<true>(sh, row, n, shift, bins, prefix, pmask);
    take_digit(sh, sh.hist, bins, shift, prefix, pmask, rem);
  }
  const uint32_t T = prefix;      // the K-th largest key
  const uint32_t R = rem;         // keys equal to T that are taken (the first R in position order)

  // ---- compaction in position order: an element's slot = (greater keys before it) +
  // min(keys equal to T before it, R)
  uint32_t gt_run = 0, tie_run = 0;
#pragma unroll 1
  for (int64_t base = 0; base < n; base += kTkGroup) {
    uint32_t k[kTkPer];
    const int64_t p0 = base + (int64_t)t * kTkPer;
    const uint32_t valid = load_keys(row, p0, n, k);
    uint32_t g = 0, e = 0;
#pragma unroll
    for (int i = 0; i < kTkPer; ++i) {
      const bool in = (valid >> i) & 1u;
      g += (in && k[i] > T) ? 1u : 0u;
      e += (in && k[i] == T) ? 1u : 0u;
    }
    uint32_t tot;
    const uint32_t ex = block_exclusive_scan(g | (e << 16), sh.warp_sums, &tot);
    uint32_t gb = gt_run + (ex & 0xFFFFu), eb = tie_run + (ex >> 16);
#pragma unroll
    for (int i = 0; i < kTkPer; ++i) {
      if (!((valid >> i) & 1u)) continue;
      if (k[i] > T) {
        o[gb + (eb < R ? eb : R)] = (int32_t)(p0 + i);
        ++gb;
      } else if (k[i] == T) {
        if (eb < R) o[gb + eb] = (int32_t)(p0 + i);
        ++eb;
      }
    }
    gt_run += tot & 0xFFFFu;
    tie_run += tot >> 16;
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* seq_lens, int B, int Q, int K,
                        int32_t* out, cudaStream_t stream) {
  // the shared-memory opt-in is per device; set it once for each device that launches
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= kMaxDevices || !done[dev]) {
      err = cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(TopkShared));
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)sizeof(TopkShared));
      if (err != cudaSuccess) return err;
      if (dev >= 0 && dev < kMaxDevices) done[dev] = true;
    }
  }
  // Rows that leave SMs idle are split over a cluster of C CTAs (C <= 8, the portable cluster size):
  // C = the SMs per row, so one wave of clusters covers the batch.
  const int64_t rows = (int64_t)B * Q;
  const int sms = device_sm_count();
  int64_t c = sms > 0 ? sms / rows : 1;
  if (c > 8) c = 8;
  if (c < 2) {
    topk_kernel<false><<<(unsigned)rows, kTkThreads, sizeof(TopkShared), stream>>>(logits, stride, seq_lens, Q, K, out,
                                                                                   1);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * c), 1, 1);
  cfg.blockDim = dim3(kTkThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(TopkShared);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel<true>, logits, stride, seq_lens, Q, K, out, (int)c);
}

}  // namespace nvfp4mla
