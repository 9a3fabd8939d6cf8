// mla_kv_pack kernel: bf16 latent + rope rows -> 352-byte NVFP4 rows in 64-token pages.
//
// Row format ("Prime Inference", translated page, "Making room for low-latency
// decode"; byte split from "Serving GLM-5.3 ...", "Four bits per latent value:
// where 352 comes from"): 256 bytes of e2m1 codes (element 2i in the low
// nibble of byte i), 32 E4M3 block scales (one per 16 latent values), 64 E4M3
// rope bytes.
//
// One warp per row, two rows per warp in flight: every load of both rows (slot,
// latent, rope) is issued before any is used, so a row costs one memory round
// trip, not a slot load followed by the data loads. Lane l loads latent
// elements 8l..8l+7 and 256+8l..256+8l+7 (two 16-byte loads; the warp reads
// the 1 KB latent row fully coalesced) and rope elements 2l, 2l+1. A 16-value
// block spans a lane pair, so one shuffle gives the block amax. The row is
// assembled in shared memory and written with 22 coalesced 16-byte stores.
// Inputs and the cache rows are streamed (read or written once).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4mla {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// e2m1 code of x for a block whose decoded scale is s: nearest grid point of
// |x|/s, ties to the even code, saturating at 6, sign bit kept. Decided
// without dividing: |x|/s vs a midpoint m is |x| vs m*s. Ties at 0.25, 1.25, 2.5, 5 go
// down (even codes 0, 2, 4, 6); ties at 0.75, 1.75, 3.5 go up (codes 2, 4, 6).
// The thresholds increase and each crossing test is monotonic in |x|, so the
// code (the number of thresholds crossed) is found by binary search: three
// compares instead of seven. The search runs on bf16 pairs (two values per
// instruction): x is bf16 and every threshold m*s has at most 7 significant
// bits (s >= 2^-9), so it is exact in bf16 and the comparisons are exact. NaN
// magnitudes cross none (code 0).
struct Thresholds {
  uint32_t t0, t1, t2, t3;               // m*s for m = 0.25, 0.75, 1.25, 1.75, as bf16 pairs
  uint32_t d51, d40, d62;                // t5 - t1, t4 - t0, t6 - t2 (0 when s = 0)
};
__device__ __forceinline__ uint32_t bf16_pair(float f) {
  const uint32_t b = __float_as_uint(f) >> 16;   // exact for E4M3 values: their low 16 bits are zero
  return b | (b << 16);
}
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) { return *reinterpret_cast<const __nv_bfloat162*>(&u); }
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) { return *reinterpret_cast<const uint32_t*>(&v); }
// Thresholds m*s and the differences between the ones a search level chooses from, two lanes per
// bf16 multiply: s (an E4M3 value, <= 4 significant bits) is exact in bf16 and so is every product
// (m and the differences 2.75, 2.25, 3.75 have <= 4 bits; products within [2^-11, 2240]). A zero
// scale makes the thresholds +inf (every finite magnitude codes 0) and the differences 0.
__device__ __forceinline__ Thresholds make_thresholds(float s) {
  const __nv_bfloat162 s2 = as_bf2(s > 0.f ? bf16_pair(s) : 0x7F807F80u);
  const __nv_bfloat162 sd = as_bf2(s > 0.f ? bf16_pair(s) : 0u);
  Thresholds t;   // bf16 pairs of 0.25, 0.75, 1.25, 1.75 and of 2.75, 2.25, 3.75
  t.t0 = as_u32(__hmul2(s2, as_bf2(0x3E803E80u))); t.t1 = as_u32(__hmul2(s2, as_bf2(0x3F403F40u)));
  t.t2 = as_u32(__hmul2(s2, as_bf2(0x3FA03FA0u))); t.t3 = as_u32(__hmul2(s2, as_bf2(0x3FE03FE0u)));
  t.d51 = as_u32(__hmul2(sd, as_bf2(0x40304030u))); t.d40 = as_u32(__hmul2(sd, as_bf2(0x40104010u)));
  t.d62 = as_u32(__hmul2(sd, as_bf2(0x40704070u)));
  return t;
}
// e2m1 codes (with sign bits) of the bf16 pair w, one per half: the element in bits 0..15 gives
// the nibble in bits 0..3, the element in bits 16..31 the nibble in bits 16..19. The search runs
// in bf16 arithmetic (the fused multiply-add pipe): each test gives 1.0 or 0.0 per half, a level's
// threshold is chosen as t_lo + g * (t_hi - t_lo) (exact: one of the two exact values), and the
// code is summed onto 128 (bf16 128 + c has c in its low mantissa bits, so c = bits ^ 0x4300).
__device__ __forceinline__ uint32_t e2m1_pair(uint32_t w, const Thresholds& t) {
  const __nv_bfloat162 a = as_bf2(w & 0x7FFF7FFFu);
  const __nv_bfloat162 g2 = __hge2(a, as_bf2(t.t3));                                   // codes 4..7
  const __nv_bfloat162 g1 = __hge2(a, __hfma2(g2, as_bf2(t.d51), as_bf2(t.t1)));       // t5 / t1
  const __nv_bfloat162 u = __hfma2(g2, as_bf2(t.d40), as_bf2(t.t0));                  // t4 / t0
  const __nv_bfloat162 v = __hfma2(g2, as_bf2(t.d62), as_bf2(t.t2));                  // t6 / t2
  const __nv_bfloat162 g0 = __hgt2(a, __hfma2(g1, __hsub2(v, u), u));
  const __nv_bfloat162 c = __hfma2(g2, as_bf2(0x40804080u), __hfma2(g1, as_bf2(0x40004000u),
                                                                     __hadd2(g0, as_bf2(0x43004300u))));
  return (as_u32(c) ^ 0x43004300u) | ((w >> 12) & 0x00080008u);
}
// 8 bf16 (one uint4) -> 8 nibbles (one 32-bit word), element 0 in bits 0..3: each pair folds its
// two nibbles into its low byte (c | c >> 12), and byte permutes gather the four bytes.
__device__ __forceinline__ uint32_t encode8(const uint4& v, const Thresholds& t) {
  const uint32_t c0 = e2m1_pair(v.x, t), c1 = e2m1_pair(v.y, t), c2 = e2m1_pair(v.z, t), c3 = e2m1_pair(v.w, t);
  const uint32_t x0 = c0 | (c0 >> 12), x1 = c1 | (c1 >> 12), x2 = c2 | (c2 >> 12), x3 = c3 | (c3 >> 12);
  return __byte_perm(__byte_perm(x0, x1, 0x0040), __byte_perm(x2, x3, 0x0040), 0x5410);
}
// max |x| of 8 bf16 (exact: bf16 abs and max, two lanes per instruction; a NaN loses to the other
// operand, as with fmaxf)
__device__ __forceinline__ float amax8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  __nv_bfloat162 m = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[0]));
#pragma unroll
  for (int i = 1; i < 4; ++i) m = __hmax2(m, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[i])));
  return fmaxf(fmaxf(__low2float(m), __high2float(m)), 0.f);
}
// The two E4M3 scale bytes of sc (byte 0, byte 1) as floats, one conversion for both.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t sc) {
  const uint32_t h2 = ptx::e4m3x2_to_f16x2(sc & 0xFFFFu);
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

constexpr int kRowsPerWarp = 2;

// RN32(1/6) = (1/6)(1 + 2^-25). For a bf16 amax, amax * RN32(1/6) rounds to the same E4M3 value as
// the exact amax/6: where amax/6 is an E4M3 rounding midpoint (at most 5 significant bits) the
// product is within 2^-25 relative of it, less than half an fp32 ulp, so it rounds onto the
// midpoint and the E4M3 rounding breaks the tie as for the exact quotient; every other amax/6 is
// at least ~2^-8 relative away from a midpoint. (Checked against the exact quotient for every
// non-negative bf16, +inf included.)
constexpr float kRcp6 = 0.16666667163372040f;   // 0x3E2AAAAB

__global__ void __launch_bounds__(kWarpsPerBlock * 32, 4) pack_kernel(
    const uint16_t* __restrict__ latent, int64_t lstride, const uint16_t* __restrict__ rope, int64_t rstride,
    const int64_t* __restrict__ slots, int64_t n, uint8_t* __restrict__ cache, int64_t num_pages,
    int32_t* __restrict__ status) {
  __shared__ __align__(16) uint8_t stage[kWarpsPerBlock][kRowsPerWarp][kRowBytes];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nslots = num_pages * kPageTokens;
  for (int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerBlock + warp) * kRowsPerWarp; row0 < n;
       row0 += (int64_t)gridDim.x * kWarpsPerBlock * kRowsPerWarp) {
    int64_t slot_v[kRowsPerWarp];
    uint4 a_v[kRowsPerWarp], b_v[kRowsPerWarp];
    uint32_t r_v[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int64_t row = row0 + i;
      const bool in = row < n;
      const uint16_t* lp = latent + (in ? row : 0) * lstride;
      slot_v[i] = in ? __ldcs(slots + row) : -1;
      a_v[i] = in ? __ldcs(reinterpret_cast<const uint4*>(lp) + lane) : make_uint4(0u, 0u, 0u, 0u);         // 8l..8l+7
      b_v[i] = in ? __ldcs(reinterpret_cast<const uint4*>(lp + 256) + lane) : make_uint4(0u, 0u, 0u, 0u);   // 256+8l..
      r_v[i] = in ? __ldcs(reinterpret_cast<const unsigned int*>(rope + row * rstride) + lane) : 0u;
    }
    // Both rows are encoded as straight-line code (a row whose slot is skipped is encoded too
    // and not stored), so the two rows' arithmetic can interleave.
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      uint8_t* srow = stage[warp][i];
      const uint4 a = a_v[i], b = b_v[i];
      const uint32_t r = r_v[i];

      // block amax: blocks (l>>1) and 16+(l>>1) span lanes 2m, 2m+1
      float ma = amax8(a), mb = amax8(b);
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      // scale = E4M3_rn_sat(amax / 6), amax/6 formed as amax * RN32(1/6) (see kRcp6)
      const uint32_t sc = ptx::f32x2_to_e4m3x2(__fmul_rn(ma, kRcp6), __fmul_rn(mb, kRcp6));
      const float2 s = e4m3x2_to_f32x2(sc);
      const Thresholds ta = make_thresholds(s.x);
      const Thresholds tb = make_thresholds(s.y);
      const uint32_t wa = encode8(a, ta), wb = encode8(b, tb);
      const uint32_t rr = ptx::bf16x2_to_e4m3x2(r);   // NaN keeps its sign (0x7F / 0xFF)

      *reinterpret_cast<uint32_t*>(srow + 4 * lane) = wa;
      *reinterpret_cast<uint32_t*>(srow + 128 + 4 * lane) = wb;
      if ((lane & 1) == 0) {
        srow[kScaleOff + (lane >> 1)] = (uint8_t)(sc & 0xFFu);
        srow[kScaleOff + 16 + (lane >> 1)] = (uint8_t)(sc >> 8);
      }
      *reinterpret_cast<uint16_t*>(srow + kRopeOff + 2 * lane) = (uint16_t)rr;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int64_t slot = slot_v[i];
      if (slot < 0 || slot >= nslots) {
        if (slot != -1 && lane == 0 && status != nullptr) atomicAdd(status + 3, 1);
        continue;
      }
      if (lane < kRowBytes / 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(stage[warp][i] + 16 * lane);
        __stcs(reinterpret_cast<uint4*>(cache + slot * kRowBytes + 16 * lane), v);
      }
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_pack(const uint16_t* latent, int64_t lstride, const uint16_t* rope, int64_t rstride,
                        const int64_t* slots, int64_t n, uint8_t* cache, int64_t num_pages, int32_t* status,
                        cudaStream_t stream) {
  const int sms = device_sm_count();
  // one resident wave of blocks, each striding over the rows (the occupancy is the same on every
  // device of this build's architecture; concurrent first calls store the same value)
  static std::atomic<int> cached_per_sm{0};
  int per_sm = cached_per_sm.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pack_kernel, kWarpsPerBlock * 32, 0) != cudaSuccess ||
        per_sm < 1) {
      (void)cudaGetLastError();
      per_sm = 2;
    }
    cached_per_sm.store(per_sm, std::memory_order_relaxed);
  }
  const int64_t want = (n + kWarpsPerBlock * kRowsPerWarp - 1) / (kWarpsPerBlock * kRowsPerWarp);
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * per_sm;
  const int grid = (int)(want < cap ? want : cap);
  pack_kernel<<<grid, kWarpsPerBlock * 32, 0, stream>>>(latent, lstride, rope, rstride, slots, n, cache,
                                                         num_pages, status);
  return cudaGetLastError();
}

}  // namespace nvfp4mla
