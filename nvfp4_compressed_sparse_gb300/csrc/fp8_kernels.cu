// Kernels of the FP8 comparison paths: the 576-byte FP8 row pack, the per-token FP8 row pack and
// the staged NVFP4 -> FP8 copy.
//
// What they compute ("Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", sections
// "Four bits per latent value: where 352 comes from" and "A kernel that reads four bits directly";
// "Prime Inference", translated page, "Native NVFP4 sparse MLA decode kernel"): an FP8 cache row is
// one E4M3 byte per value of the 576-value row (512 latent + 64 rope); the staged path reads each
// selected 352-byte NVFP4 row and writes a 576-byte FP8 copy that an FP8 attention kernel then
// reads (1,504 bytes per selected row through HBM, against 352 for the native kernel).
//
// Roundings (this build's readings): E4M3 nearest-even, saturating at +-448, NaN -> 0x7F with its
// sign; a staged latent value is e2m1(code) * E4M3(scale), exact in fp16, rounded once; a block with
// a NaN scale byte stages as 0x7F; rope bytes are copied.
//
// The pack is one warp per row; the staging resolves 32 entries per warp at once and copies their
// rows four at a time. Every load of a row is issued before any is used; stores are 16-byte
// coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4mla {
namespace {

constexpr int kFp8Warps = 8;   // warps per block of either kernel

// bf16 rows -> FP8 rows. Lane l converts latent values 16l..16l+15 (two 16-byte loads; the warp
// reads the 1 KB latent row coalesced) and rope values 2l, 2l+1.
__global__ void __launch_bounds__(kFp8Warps * 32) fp8_pack_kernel(
    const uint16_t* __restrict__ latent, int64_t lstride, const uint16_t* __restrict__ rope, int64_t rstride,
    const int64_t* __restrict__ slots, int64_t n, uint8_t* __restrict__ cache, int64_t num_pages,
    int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t nslots = num_pages * kPageTokens;
  for (int64_t row = (int64_t)blockIdx.x * kFp8Warps + (threadIdx.x >> 5); row < n;
       row += (int64_t)gridDim.x * kFp8Warps) {
    const int64_t slot = __ldcs(slots + row);
    const uint4* lp = reinterpret_cast<const uint4*>(latent + row * lstride) + 2 * lane;
    const uint4 a = __ldcs(lp), b = __ldcs(lp + 1);
    const uint32_t r = __ldcs(reinterpret_cast<const unsigned int*>(rope + row * rstride) + lane);
    if (slot < 0 || slot >= nslots) {
      if (slot != -1 && lane == 0 && status != nullptr) atomicAdd(status + 3, 1);
      continue;
    }
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = ptx::bf16x2_to_e4m3x2(w[2 * i]) | (ptx::bf16x2_to_e4m3x2(w[2 * i + 1]) << 16);
    uint8_t* dst = cache + slot * kFp8RowBytes;
    __stcs(reinterpret_cast<uint4*>(dst) + lane, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(reinterpret_cast<unsigned short*>(dst + kLatent) + lane, (unsigned short)ptx::bf16x2_to_e4m3x2(r));
  }
}

// bf16 rows -> per-token FP8 rows (672 bytes: E4M3 latent / scale, bf16 rope / scale, fp32 scale,
// zero padding), the arithmetic of TokenSpeed's per-token write path: amax over the 512 latent
// values, scale = max(amax, 1e-26) / 448, both divisions in IEEE fp32 (round to nearest even),
// E4M3 (nearest even, saturating) and bf16 (nearest even) rounding. Lane l holds latent values
// 16l..16l+15 and rope values 2l, 2l+1. Finite inputs (a NaN or an infinity gives an unspecified
// row).
__global__ void __launch_bounds__(kFp8Warps * 32) token_pack_kernel(
    const uint16_t* __restrict__ latent, int64_t lstride, const uint16_t* __restrict__ rope, int64_t rstride,
    const int64_t* __restrict__ slots, int64_t n, uint8_t* __restrict__ cache, int64_t num_pages,
    int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int64_t nslots = num_pages * kPageTokens;
  for (int64_t row = (int64_t)blockIdx.x * kFp8Warps + (threadIdx.x >> 5); row < n;
       row += (int64_t)gridDim.x * kFp8Warps) {
    const int64_t slot = __ldcs(slots + row);
    const uint4* lp = reinterpret_cast<const uint4*>(latent + row * lstride) + 2 * lane;
    const uint4 a = __ldcs(lp), b = __ldcs(lp + 1);
    const uint32_t r = __ldcs(reinterpret_cast<const unsigned int*>(rope + row * rstride) + lane);
    if (slot < 0 || slot >= nslots) {
      if (slot != -1 && lane == 0 && status != nullptr) atomicAdd(status + 3, 1);
      continue;
    }
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float x[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(fmaxf(amax, 1e-26f), 448.0f);
    uint32_t o4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o4[i] = ptx::f32x2_to_e4m3x2(__fdiv_rn(x[4 * i], scale), __fdiv_rn(x[4 * i + 1], scale)) |
              (ptx::f32x2_to_e4m3x2(__fdiv_rn(x[4 * i + 2], scale), __fdiv_rn(x[4 * i + 3], scale)) << 16);
    const __nv_bfloat162 rb = __floats2bfloat162_rn(__fdiv_rn(__uint_as_float(r << 16), scale),
                                                    __fdiv_rn(__uint_as_float(r & 0xFFFF0000u), scale));
    uint8_t* dst = cache + slot * kTokRowBytes;
    __stcs(reinterpret_cast<uint4*>(dst) + lane, make_uint4(o4[0], o4[1], o4[2], o4[3]));
    __stcs(reinterpret_cast<unsigned int*>(dst + kTokRopeOff) + lane, *reinterpret_cast<const unsigned int*>(&rb));
    if (lane < 2)
      __stcs(reinterpret_cast<uint4*>(dst + kTokScaleOff) + lane,
             make_uint4(lane == 0 ? __float_as_uint(scale) : 0u, 0u, 0u, 0u));
  }
}

// FP8 copy of one NVFP4 row: lane l stages latent block l (8 nibble bytes, scale byte sc) into
// 16 E4M3 bytes; lanes 0..3 carry 16 rope bytes each (rp).
__device__ __forceinline__ uint4 stage_block(uint2 nib, uint32_t sc) {
  if ((sc & 0x7Fu) == 0x7Fu) return make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);   // NaN scale
  const uint32_t s2 = ptx::e4m3x2_to_f16x2(sc | (sc << 8));   // (scale, scale), exact
  uint32_t c0[4], c1[4];   // values 0..7 and 8..15 of the block as f16 pairs
  ptx::e2m1x8_to_f16x2x4(nib.x, c0);
  ptx::e2m1x8_to_f16x2x4(nib.y, c1);
  // products e2m1 x E4M3 have at most 5 significant bits and lie within [2^-10, 2688]: exact in fp16
  uint4 o;
  o.x = ptx::f16x2_to_e4m3x2(ptx::hmul2(c0[0], s2)) | (ptx::f16x2_to_e4m3x2(ptx::hmul2(c0[1], s2)) << 16);
  o.y = ptx::f16x2_to_e4m3x2(ptx::hmul2(c0[2], s2)) | (ptx::f16x2_to_e4m3x2(ptx::hmul2(c0[3], s2)) << 16);
  o.z = ptx::f16x2_to_e4m3x2(ptx::hmul2(c1[0], s2)) | (ptx::f16x2_to_e4m3x2(ptx::hmul2(c1[1], s2)) << 16);
  o.w = ptx::f16x2_to_e4m3x2(ptx::hmul2(c1[2], s2)) | (ptx::f16x2_to_e4m3x2(ptx::hmul2(c1[3], s2)) << 16);
  return o;
}

constexpr int kStageRowsInFlight = 4;

// A warp takes 32 consecutive (query, list entry) pairs of a decode step. Lane l resolves entry
// e0 + l with the decode's rule (the index, then its page-table word: all 32 in flight at once)
// and writes the staged decode's list entry (i or -1). The warp then copies the usable rows,
// kStageRowsInFlight at a time with every load of a group issued before any is used: lane l
// stages latent block l of each row, lanes 0..3 copy its 64 rope bytes. Also writes the staged
// decode's identity page table and lengths.
__global__ void __launch_bounds__(kFp8Warps * 32) stage_kernel(
    const uint8_t* __restrict__ cache, int64_t num_pages, const int32_t* __restrict__ page_table, int64_t max_pages,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ seq_lens, int Q, int K, int64_t entries,
    uint8_t* __restrict__ staged, int32_t* __restrict__ staged_idx, int32_t* __restrict__ staged_pt,
    int32_t* __restrict__ staged_sl, int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int pages_per_unit = K / kPageTokens;
  for (int64_t e0 = ((int64_t)blockIdx.x * kFp8Warps + (threadIdx.x >> 5)) * 32; e0 < entries;
       e0 += (int64_t)gridDim.x * kFp8Warps * 32) {
    const int64_t e = e0 + lane;
    const bool live = e < entries;
    const int64_t u = live ? e / K : 0;
    const int i = (int)(e - u * K);
    const int b = (int)(u / Q), j = (int)(u - (int64_t)b * Q);
    if (live && i < pages_per_unit) staged_pt[u * pages_per_unit + i] = (int32_t)(u * pages_per_unit + i);
    if (live && i == 0) staged_sl[u] = K;
    const int L = live ? __ldg(seq_lens + b) : 0;
    const int x = live ? __ldcs(idx + e) : -1;
    const bool in_range = x >= 0 && x < L && x <= L - Q + j;
    const bool col_ok = in_range && (int64_t)(x >> 6) < max_pages;
    const int page = col_ok ? __ldg(page_table + (int64_t)b * max_pages + (x >> 6)) : -1;
    const bool ok = col_ok && page >= 0 && page < num_pages;
    if (live) {
      staged_idx[e] = ok ? i : -1;
      if (status != nullptr) {
        if (x != -1 && !in_range) atomicAdd(status + 0, 1);
        if (in_range && !ok) atomicAdd(status + 1, 1);
      }
    }
    const int64_t row_off = ok ? ((int64_t)page * kPageTokens + (x & 63)) * kRowBytes : -1;
    uint32_t todo = __ballot_sync(0xffffffffu, ok);
    while (todo != 0u) {
      int src[kStageRowsInFlight];
      const uint8_t* row[kStageRowsInFlight];
#pragma unroll
      for (int r = 0; r < kStageRowsInFlight; ++r) {
        src[r] = todo != 0u ? __ffs(todo) - 1 : -1;
        if (todo != 0u) todo &= todo - 1u;
        const int64_t off = __shfl_sync(0xffffffffu, row_off, src[r] < 0 ? 0 : src[r]);
        row[r] = src[r] < 0 ? nullptr : cache + off;
      }
      uint2 nib[kStageRowsInFlight];
      uint32_t sc[kStageRowsInFlight];
      uint4 rp[kStageRowsInFlight];
#pragma unroll
      for (int r = 0; r < kStageRowsInFlight; ++r) {
        if (row[r] == nullptr) continue;
        nib[r] = __ldcs(reinterpret_cast<const uint2*>(row[r]) + lane);
        sc[r] = __ldcs(row[r] + kScaleOff + lane);
        if (lane < 4) rp[r] = __ldcs(reinterpret_cast<const uint4*>(row[r] + kRopeOff) + lane);
      }
#pragma unroll
      for (int r = 0; r < kStageRowsInFlight; ++r) {
        if (row[r] == nullptr) continue;
        uint8_t* dst = staged + (e0 + src[r]) * kFp8RowBytes;
        __stcs(reinterpret_cast<uint4*>(dst) + lane, stage_block(nib[r], sc[r]));
        if (lane < 4) __stcs(reinterpret_cast<uint4*>(dst + kLatent) + lane, rp[r]);
      }
    }
  }
}

int blocks_for(int64_t warps_needed, const void* kernel) {
  const int sms = device_sm_count();
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFp8Warps * 32, 0) != cudaSuccess || per_sm < 1) {
    (void)cudaGetLastError();
    per_sm = 4;
  }
  const int64_t want = (warps_needed + kFp8Warps - 1) / kFp8Warps;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * per_sm;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_fp8_pack(const uint16_t* latent, int64_t lstride, const uint16_t* rope, int64_t rstride,
                            const int64_t* slots, int64_t n, uint8_t* cache, int64_t num_pages, int32_t* status,
                            cudaStream_t stream) {
  const int grid = blocks_for(n, (const void*)fp8_pack_kernel);
  fp8_pack_kernel<<<grid, kFp8Warps * 32, 0, stream>>>(latent, lstride, rope, rstride, slots, n, cache, num_pages,
                                                       status);
  return cudaGetLastError();
}

cudaError_t launch_token_pack(const uint16_t* latent, int64_t lstride, const uint16_t* rope, int64_t rstride,
                              const int64_t* slots, int64_t n, uint8_t* cache, int64_t num_pages, int32_t* status,
                              cudaStream_t stream) {
  const int grid = blocks_for(n, (const void*)token_pack_kernel);
  token_pack_kernel<<<grid, kFp8Warps * 32, 0, stream>>>(latent, lstride, rope, rstride, slots, n, cache,
                                                         num_pages, status);
  return cudaGetLastError();
}

cudaError_t launch_stage(const uint8_t* cache, int64_t num_pages, const int32_t* page_table, int64_t max_pages,
                         const int32_t* idx, const int32_t* seq_lens, int B, int Q, int K, uint8_t* staged,
                         int32_t* staged_idx, int32_t* staged_pt, int32_t* staged_sl, int32_t* status,
                         cudaStream_t stream) {
  const int64_t entries = (int64_t)B * Q * K;
  const int grid = blocks_for((entries + 31) / 32, (const void*)stage_kernel);
  stage_kernel<<<grid, kFp8Warps * 32, 0, stream>>>(cache, num_pages, page_table, max_pages, idx, seq_lens, Q, K,
                                                     entries, staged, staged_idx, staged_pt, staged_sl, status);
  return cudaGetLastError();
}

}  // namespace nvfp4mla
