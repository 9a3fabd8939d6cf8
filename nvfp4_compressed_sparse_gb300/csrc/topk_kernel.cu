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
// GB300 design: one 1024-thread CTA per query row, an exact radix select on order-preserving
// 32-bit keys. Three histogram sweeps (key bits 31..20, 19..8, 7..0, each over the keys that
// match the digits found so far) find the threshold key T and how many keys equal to T are
// taken; one compaction sweep writes the positions. Every sweep is coalesced: a thread owns 8
// consecutive positions (two 16-byte loads), a warp 1 KB of the row, and two such groups are in
// flight per thread. The compaction keeps position order with one block-wide scan of packed
// (greater, tie) counts per 8,192 positions.
#include <cuda_runtime.h>

#include "internal.h"

namespace nvfp4mla {
namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkPer = 8;                        // consecutive positions per thread per group
constexpr int kTkGroup = kTkThreads * kTkPer;    // positions per group (8,192)

// Unsigned order of the key = selection order of the float (NaN lowest, -0.0 below +0.0).
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  if ((bits & 0x7FFFFFFFu) > 0x7F800000u) return 0u;   // NaN
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Keys of positions p0..p0+7 of the row; positions >= n get key 0 and valid = 0.
__device__ __forceinline__ uint32_t load_keys(const float* row, int64_t p0, int64_t n, uint32_t (&k)[kTkPer]) {
  if (p0 + kTkPer <= n) {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(row + p0));
    const uint4 b = __ldcs(reinterpret_cast<const uint4*>(row + p0) + 1);
    k[0] = order_key(a.x); k[1] = order_key(a.y); k[2] = order_key(a.z); k[3] = order_key(a.w);
    k[4] = order_key(b.x); k[5] = order_key(b.y); k[6] = order_key(b.z); k[7] = order_key(b.w);
    return 0xFFu;
  }
  uint32_t valid = 0;
#pragma unroll
  for (int i = 0; i < kTkPer; ++i) {
    const bool in = p0 + i < n;
    k[i] = in ? order_key(__float_as_uint(__ldcs(row + p0 + i))) : 0u;
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
  uint32_t hist[4096];
  uint32_t warp_sums[32];
  uint32_t found_digit, found_rem;
};

__global__ void __launch_bounds__(kTkThreads, 1) topk_kernel(const float* __restrict__ logits, int64_t stride,
                                                             const int32_t* __restrict__ seq_lens, int Q, int K,
                                                             int32_t* __restrict__ out) {
  __shared__ TopkShared sh;
  const int64_t rowi = blockIdx.x;
  const int b = (int)(rowi / Q), j = (int)(rowi - (int64_t)b * Q);
  int64_t n = (int64_t)__ldg(seq_lens + b) - Q + j + 1;
  if (n < 0) n = 0;
  if (n > stride) n = stride;
  int32_t* o = out + rowi * K;
  const int t = threadIdx.x;
  if (n <= K) {   // the whole range is selected
    for (int i = t; i < K; i += kTkThreads) o[i] = i < n ? i : -1;
    return;
  }
  const float* row = logits + rowi * stride;

  // ---- radix select of the K-th largest key: digits of 12, 12 and 8 bits
  uint32_t prefix = 0, pmask = 0;
  uint32_t rem = (uint32_t)K;   // rank (from the top) of the wanted key among those matching prefix
#pragma unroll 1
  for (int d = 0; d < 3; ++d) {
    const int shift = d == 0 ? 20 : (d == 1 ? 8 : 0), bins = d < 2 ? 4096 : 256;
    for (int i = t; i < bins; i += kTkThreads) sh.hist[i] = 0;
    __syncthreads();
#pragma unroll 1
    for (int64_t base = 0; base < n; base += 2 * kTkGroup) {
      uint32_t k0[kTkPer], k1[kTkPer];
      const uint32_t v0 = load_keys(row, base + (int64_t)t * kTkPer, n, k0);
      const uint32_t v1 = load_keys(row, base + kTkGroup + (int64_t)t * kTkPer, n, k1);
#pragma unroll
      for (int i = 0; i < kTkPer; ++i) {
        if (((v0 >> i) & 1u) && (k0[i] & pmask) == prefix) atomicAdd(&sh.hist[(k0[i] >> shift) & (bins - 1)], 1u);
        if (((v1 >> i) & 1u) && (k1[i] & pmask) == prefix) atomicAdd(&sh.hist[(k1[i] >> shift) & (bins - 1)], 1u);
      }
    }
    __syncthreads();
    // bins are scanned from the top: thread t owns bins [bins - per*(t+1), bins - per*t)
    const int per = bins / kTkThreads > 0 ? bins / kTkThreads : 1;
    const int hi = bins - per * t;          // exclusive upper end of this thread's bins
    uint32_t mine = 0;
    if (hi > 0)
      for (int i = 1; i <= per; ++i) mine += sh.hist[hi - i];
    uint32_t total;
    const uint32_t above = block_exclusive_scan(mine, sh.warp_sums, &total);   // counts in higher bins
    if (hi > 0 && above < rem && above + mine >= rem) {
      uint32_t cum = above;
      for (int i = 1; i <= per; ++i) {
        const uint32_t h = sh.hist[hi - i];
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
  topk_kernel<<<(unsigned)((int64_t)B * Q), kTkThreads, 0, stream>>>(logits, stride, seq_lens, Q, K, out);
  return cudaGetLastError();
}

}  // namespace nvfp4mla
