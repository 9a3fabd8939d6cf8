// Host side of the C ABI declared in include/nvfp4mla.h: argument checks,
// work split, workspace carving and kernel launches. No allocation, no
// synchronisation; everything is enqueued on the caller's stream.
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <mutex>

#include "../../include/nvfp4mla.h"
#include "internal.h"

namespace nvfp4mla {

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static int cached[64] = {0};
  if (dev < 0 || dev >= 64) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) cached[dev] = n;
  }
  return cached[dev];
}

DecodeSchedule make_schedule(int B, int Q, int H, int topk, int num_sms, int max_ctas, ClusterPolicy policy) {
  DecodeSchedule s{};
  const int nh = H < kHeadsPerCta ? H : kHeadsPerCta;
  s.units = (int64_t)B * Q * (H / nh);
  s.tiles_per_unit = (topk + kTileTokens - 1) / kTileTokens;
  s.total_tiles = s.units * s.tiles_per_unit;
  int64_t g = num_sms > 0 ? num_sms : 1;
  if (max_ctas > 0 && max_ctas < g) g = max_ctas;
  if (g > s.total_tiles) g = s.total_tiles;
  s.ctas = (int)g;
  s.partial_slots = s.ctas + s.units - 1;
  s.cluster = 0;
  s.pair = 0;
  if (policy == kPairSplit) {
    // one stream-K range per pair of SMs
    int64_t pairs = num_sms > 1 ? num_sms / 2 : 1;
    if (max_ctas > 0 && max_ctas < pairs) pairs = max_ctas;
    if (pairs > s.total_tiles) pairs = s.total_tiles;
    s.ctas = (int)pairs;
    s.partial_slots = s.ctas + s.units - 1;
    s.pair = 1;
    return s;
  }
  // Cluster schedule: G = min(8, SMs / units, tiles per unit) CTAs per unit, one wave; it needs no
  // q-prep and no merge grid. kClusterBalanced takes it when no CTA then runs more tiles than under
  // the stream-K split, kClusterAny whenever G >= 1 (to measure the schedules against each other).
  // Measured on GB300 (with the two-part fp16 weights) the split was faster at every size tried:
  // 64 queries 54.2 vs 55.6 us (G = 2), 128 queries 93.9 vs 96.9 us (G = 1), 1 and 4 queries ~8 us
  // faster than 8-CTA clusters; so kClusterDefault, the policy without flags, is the split.
  if (policy != kClusterNone && max_ctas == 0 && num_sms > 0) {
    int64_t c = num_sms / s.units;
    if (c > 8) c = 8;
    if (c > s.tiles_per_unit) c = s.tiles_per_unit;
    if (c >= 1) {
      const int64_t per_cta_cluster = (s.tiles_per_unit + c - 1) / c;
      const int64_t per_cta_split = (s.total_tiles + s.ctas - 1) / s.ctas;
      const bool take = policy == kClusterAny || (policy == kClusterBalanced && per_cta_cluster <= per_cta_split);
      if (take) {
        s.cluster = (int)c;
        s.ctas = (int)(s.units * c);
      }
    }
  }
  return s;
}

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: partial O [slots, nh, 512] f32 | partial (max, sum) [slots, nh, 2] f32 |
// FP16 q images [units, 9 * nh * 128] | q scales [units] f32 | partial-ready flags [slots] u64;
// each part 256-byte aligned.
struct WorkspaceLayout {
  size_t o, ml, q16, qscale, flag, total;
};
static WorkspaceLayout layout_for(const DecodeSchedule& s, int H) {
  const int nh = H < kHeadsPerCta ? H : kHeadsPerCta;
  WorkspaceLayout w;
  w.o = 0;
  w.ml = w.o + align256((size_t)s.partial_slots * nh * kLatent * sizeof(float));
  w.q16 = w.ml + align256((size_t)s.partial_slots * nh * 2 * sizeof(float));
  w.qscale = w.q16 + align256((size_t)s.units * 9 * nh * 128);
  w.flag = w.qscale + align256((size_t)s.units * sizeof(float));
  w.total = w.flag + align256((size_t)s.partial_slots * sizeof(uint64_t));
  return w;
}

size_t workspace_bytes_for(const DecodeSchedule& s, int H) { return layout_for(s, H).total; }

static bool sizes_ok(int B, int Q, int H, int topk) {
  if (B < 1 || Q < 1 || Q > 16 || topk < 1 || topk > NVFP4MLA_MAX_TOPK) return false;
  return H == 16 || H == 32 || H == 64 || H == 128;
}

static inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Memory the decode kernels may read or write with this pointer: device or managed memory of the
// current device, or page-locked host memory mapped for the device at the same address (the
// kernels then move those bytes over the host link themselves). Anything else (pageable host
// memory, another device's memory, an unknown pointer) is invalid and rejected before any launch.
enum PtrKind { kPtrInvalid, kPtrDevice, kPtrHost };
static PtrKind pointer_kind(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return kPtrInvalid;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return kPtrInvalid;
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return a.device == dev ? kPtrDevice : kPtrInvalid;
    case cudaMemoryTypeHost:
      return a.devicePointer == p ? kPtrHost : kPtrInvalid;
    default:
      return kPtrInvalid;
  }
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The cache as a 2-D tensor of uint32: rows of row_bytes / 4 words (88 for the 352-byte NVFP4 row,
// 144 for the 576-byte FP8 row), one row per token slot. Row gathers use TMA tile::gather4 with a
// one-row box; rows outside [0, rows) (the -1 of unused entries) read as zeros.
static bool encode_cache_map(CUtensorMap* map, const void* cache, int64_t num_pages, int row_bytes) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)(num_pages * kPageTokens)};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(row_bytes / 4), 1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace nvfp4mla

using namespace nvfp4mla;

// A tag no earlier call of this process used (odd, so never 0): the merge grid recognises the
// partials of this call by it, so the workspace needs no clearing between calls.
static uint64_t next_call_tag() {
  static std::atomic<uint64_t> counter{0};
  static const uint64_t seed = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
  uint64_t z = seed + 0x9E3779B97F4A7C15ull * (counter.fetch_add(1, std::memory_order_relaxed) + 1);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;   // splitmix64 finaliser
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return (z ^ (z >> 31)) | 1ull;
}

// The decode grid for these sizes and flags on the current device: the stream-K split unless a
// cluster flag makes make_schedule pick the cluster schedule and all its clusters can be resident
// at once. (With results in host memory the split's merge grid streams them over the host link as
// units finish; host_results keeps it there unless a cluster flag is given.)
static bool plan_on_device(int B, int Q, int H, int topk, uint32_t flags, bool host_results, DecodeSchedule* out) {
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  ClusterPolicy policy = host_results ? kClusterNone : kClusterDefault;
  if (flags & NVFP4MLA_FLAG_CLUSTER) policy = (flags & NVFP4MLA_FLAG_CLUSTER_ANY) ? kClusterAny : kClusterBalanced;
  if (flags & NVFP4MLA_FLAG_SPLIT) policy = kClusterNone;
  if ((flags & NVFP4MLA_FLAG_PAIR) && !host_results && !(flags & NVFP4MLA_FLAG_SPLIT)) policy = kPairSplit;
  DecodeSchedule s = make_schedule(B, Q, H, topk, sms, (int)(flags & 0xFFFFu), policy);
  if (s.pair && max_active_pairs(H < kHeadsPerCta ? H : kHeadsPerCta) < s.ctas)
    s = make_schedule(B, Q, H, topk, sms, (int)(flags & 0xFFFFu), kClusterNone);
  if (s.cluster > 1) {
    const int fit = max_active_clusters(H < kHeadsPerCta ? H : kHeadsPerCta, s.cluster);
    if (fit < s.units) s = make_schedule(B, Q, H, topk, sms, (int)(flags & 0xFFFFu), kClusterNone);
  }
  *out = s;
  return true;
}

namespace nvfp4mla {
// Workspace bytes sparse_mla_decode needs for these sizes and flags on the current device, with the
// same checks and return codes as the call itself (OK, INVALID_ARG, UNSUPPORTED, CUDA).
int decode_workspace_need(int B, int Q, int H, int topk, uint32_t flags, size_t* need) {
  if (!sizes_ok(B, Q, H, topk)) return NVFP4MLA_ERR_INVALID_ARG;
  DecodeSchedule s;
  if (!plan_on_device(B, Q, H, topk, flags, false, &s)) return NVFP4MLA_ERR_CUDA;
  if (s.total_tiles > (int64_t)INT32_MAX) return NVFP4MLA_ERR_UNSUPPORTED;
  *need = workspace_bytes_for(s, H);
  return NVFP4MLA_OK;
}
}  // namespace nvfp4mla

extern "C" {

const char* nvfp4mla_status_string(int status) {
  switch (status) {
    case NVFP4MLA_OK: return "ok";
    case NVFP4MLA_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4MLA_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case NVFP4MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case NVFP4MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4MLA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int mla_kv_pack(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                const int64_t* slot_mapping, int64_t num_tokens, void* kv_cache, int64_t num_pages,
                int32_t* dev_status, void* stream) {
  if (num_tokens < 0 || num_pages < 1) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return NVFP4MLA_OK;
  if (latent == nullptr || rope == nullptr || slot_mapping == nullptr || kv_cache == nullptr)
    return NVFP4MLA_ERR_INVALID_ARG;
  if (latent_row_stride < kLatent || rope_row_stride < kRope) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages > (INT64_MAX / (kPageTokens * kRowBytes))) return NVFP4MLA_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || (latent_row_stride % 8) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(rope, 4) || (rope_row_stride % 2) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(kv_cache, 16) || !aligned(slot_mapping, 8)) return NVFP4MLA_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return NVFP4MLA_ERR_ALIGNMENT;
  // The pack kernel reads and writes device memory only: pageable or page-locked host memory,
  // another device's memory or an unknown pointer is rejected before anything is enqueued.
  if (pointer_kind(latent) != kPtrDevice || pointer_kind(rope) != kPtrDevice ||
      pointer_kind(slot_mapping) != kPtrDevice || pointer_kind(kv_cache) != kPtrDevice ||
      (dev_status != nullptr && pointer_kind(dev_status) != kPtrDevice))
    return NVFP4MLA_ERR_INVALID_ARG;
  const cudaError_t err = launch_pack(static_cast<const uint16_t*>(latent), latent_row_stride,
                                      static_cast<const uint16_t*>(rope), rope_row_stride, slot_mapping,
                                      num_tokens, static_cast<uint8_t*>(kv_cache), num_pages, dev_status,
                                      static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? NVFP4MLA_OK : NVFP4MLA_ERR_CUDA;
}

int indexer_topk(const float* logits, int64_t logits_row_stride, const int32_t* seq_lens, int B, int Q, int topk,
                 int32_t* topk_indices, void* stream) {
  if (B < 1 || Q < 1 || Q > 16 || topk < 1 || topk > NVFP4MLA_MAX_TOPK) return NVFP4MLA_ERR_INVALID_ARG;
  if ((int64_t)B * Q > (int64_t)INT32_MAX) return NVFP4MLA_ERR_UNSUPPORTED;
  if (logits == nullptr || seq_lens == nullptr || topk_indices == nullptr) return NVFP4MLA_ERR_INVALID_ARG;
  if (logits_row_stride < 1 || logits_row_stride > (int64_t)INT32_MAX) return NVFP4MLA_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || (logits_row_stride % 4) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(seq_lens, 4) || !aligned(topk_indices, 4)) return NVFP4MLA_ERR_ALIGNMENT;
  if (pointer_kind(logits) != kPtrDevice || pointer_kind(seq_lens) != kPtrDevice ||
      pointer_kind(topk_indices) != kPtrDevice)
    return NVFP4MLA_ERR_INVALID_ARG;
  const cudaError_t err = launch_topk(logits, logits_row_stride, seq_lens, B, Q, topk, topk_indices,
                                      static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? NVFP4MLA_OK : NVFP4MLA_ERR_CUDA;
}

int sparse_mla_decode_plan(int B, int Q, int H, int topk, uint32_t flags, int* ctas, int* cluster) {
  if (!sizes_ok(B, Q, H, topk)) return NVFP4MLA_ERR_INVALID_ARG;
  DecodeSchedule s;
  if (!plan_on_device(B, Q, H, topk, flags, false, &s)) return NVFP4MLA_ERR_CUDA;
  if (ctas != nullptr) *ctas = s.pair ? 2 * s.ctas : s.ctas;
  if (cluster != nullptr) *cluster = s.pair ? -2 : s.cluster;
  return NVFP4MLA_OK;
}

size_t sparse_mla_decode_workspace_size(int B, int Q, int H, int topk, int num_sms) {
  if (!sizes_ok(B, Q, H, topk)) return 0;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return 0;
  const DecodeSchedule s = make_schedule(B, Q, H, topk, num_sms, 0, kClusterNone);
  if (s.total_tiles > (int64_t)INT32_MAX) return 0;
  return workspace_bytes_for(s, H);
}

}  // extern "C"

// Folded query tokens of sparse_mla_decode_shared (nullptr: none).
struct FoldArgs {
  const uint8_t* member;
  int q, h;
};

// sparse_mla_decode over either row format (row_fmt 0: 352-byte NVFP4 rows; 1, 2: FP8 rows, split
// schedule and results in device memory only), optionally with folded query tokens.
static int decode_impl(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* page_table,
                       int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens, int B, int Q,
                       int H, int topk, float softmax_scale, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, uint32_t flags, void* stream, int row_fmt,
                       const FoldArgs* fold = nullptr) {
  const int row_bytes = row_fmt == 1 ? kFp8RowBytes : (row_fmt == 2 ? kTokRowBytes : kRowBytes);
  if (!sizes_ok(B, Q, H, topk)) return NVFP4MLA_ERR_INVALID_ARG;
  if (q == nullptr || kv_cache == nullptr || page_table == nullptr || topk_indices == nullptr ||
      seq_lens == nullptr || out == nullptr || lse == nullptr)
    return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_pages_per_seq < 1) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages > (INT64_MAX / (kPageTokens * row_bytes)) || num_pages > INT32_MAX) return NVFP4MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return NVFP4MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16)) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(page_table, 4) || !aligned(topk_indices, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4))
    return NVFP4MLA_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return NVFP4MLA_ERR_ALIGNMENT;
  const PtrKind k_out = pointer_kind(out), k_lse = pointer_kind(lse);
  if (pointer_kind(q) == kPtrInvalid || pointer_kind(page_table) == kPtrInvalid ||
      pointer_kind(topk_indices) == kPtrInvalid || pointer_kind(seq_lens) == kPtrInvalid || k_out == kPtrInvalid ||
      k_lse == kPtrInvalid || pointer_kind(kv_cache) != kPtrDevice ||
      (dev_status != nullptr && pointer_kind(dev_status) != kPtrDevice))
    return NVFP4MLA_ERR_INVALID_ARG;
  if (row_fmt != 0 || fold != nullptr) {
    if (k_out != kPtrDevice || k_lse != kPtrDevice) return NVFP4MLA_ERR_UNSUPPORTED;
    flags = (flags & ~(NVFP4MLA_FLAG_CLUSTER | NVFP4MLA_FLAG_CLUSTER_ANY | NVFP4MLA_FLAG_PAIR)) | NVFP4MLA_FLAG_SPLIT;
  }
  DecodeSchedule s;
  if (!plan_on_device(B, Q, H, topk, flags, k_out == kPtrHost || k_lse == kPtrHost, &s)) return NVFP4MLA_ERR_CUDA;
  const size_t need = workspace_bytes_for(s, H);
  if (workspace == nullptr || workspace_bytes < need) return NVFP4MLA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return NVFP4MLA_ERR_ALIGNMENT;
  if (pointer_kind(workspace) != kPtrDevice) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages * kPageTokens > (int64_t)INT32_MAX) return NVFP4MLA_ERR_UNSUPPORTED;   // int32 row coordinates
  if (s.total_tiles > (int64_t)INT32_MAX) return NVFP4MLA_ERR_UNSUPPORTED;               // int32 tile numbers

  DecodeParams p{};
  if (!encode_cache_map(&p.cache_map, kv_cache, num_pages, row_bytes)) return NVFP4MLA_ERR_CUDA;
  p.row_fmt = row_fmt;
  p.q = static_cast<const uint16_t*>(q);
  p.cache = static_cast<const uint8_t*>(kv_cache);
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.max_pages = max_pages_per_seq;
  p.idx = topk_indices;
  p.seq_lens = seq_lens;
  p.B = B;
  p.Q = Q;
  p.H = H;
  p.topk = topk;
  p.heads_per_cta = H < kHeadsPerCta ? H : kHeadsPerCta;
  p.head_groups = H / p.heads_per_cta;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  const WorkspaceLayout wl = layout_for(s, H);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  p.part_o = reinterpret_cast<float*>(wsb + wl.o);
  p.part_ml = reinterpret_cast<float*>(wsb + wl.ml);
  p.q16 = wsb + wl.q16;
  p.qscale = reinterpret_cast<float*>(wsb + wl.qscale);
  p.part_flag = reinterpret_cast<uint64_t*>(wsb + wl.flag);
  p.tag = next_call_tag();
  p.merge_poll = (k_out == kPtrHost || k_lse == kPtrHost) ? 1 : 0;
  p.status = dev_status;
  p.units = s.units;
  p.total_tiles = s.total_tiles;
  p.tiles_per_unit = s.tiles_per_unit;
  p.ctas = s.ctas;
  p.cluster = s.cluster;
  p.pair = s.pair;
  p.withhold = (flags & NVFP4MLA_FLAG_TEST_TIMEOUT) ? 1u : 0u;
  p.fold_member = fold ? fold->member : nullptr;
  p.fold_q = fold ? fold->q : 1;
  p.fold_h = fold ? fold->h : H;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_decode(p, st) != cudaSuccess) return NVFP4MLA_ERR_CUDA;
  if (p.cluster == 0 && launch_merge(p, st) != cudaSuccess) return NVFP4MLA_ERR_CUDA;
  return NVFP4MLA_OK;
}

extern "C" {

int sparse_mla_decode(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* page_table,
                      int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens, int B,
                      int Q, int H, int topk, float softmax_scale, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, int32_t* dev_status, uint32_t flags, void* stream) {
  return decode_impl(q, kv_cache, num_pages, page_table, max_pages_per_seq, topk_indices, seq_lens, B, Q, H, topk,
                     softmax_scale, out, lse, workspace, workspace_bytes, dev_status, flags, stream, 0);
}

int sparse_mla_decode_fp8(const void* q, const void* kv_cache_fp8, int64_t num_pages, const int32_t* page_table,
                          int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens, int B,
                          int Q, int H, int topk, float softmax_scale, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return decode_impl(q, kv_cache_fp8, num_pages, page_table, max_pages_per_seq, topk_indices, seq_lens, B, Q, H,
                     topk, softmax_scale, out, lse, workspace, workspace_bytes, dev_status, 0u, stream, 1);
}

int sparse_mla_decode_shared(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* page_table,
                             int64_t max_pages_per_seq, const int32_t* shared_indices, const uint8_t* member_masks,
                             const int32_t* seq_lens, int B, int Q, int H, int topk, float softmax_scale, void* out,
                             float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status, uint32_t flags,
                             void* stream) {
  if (Q < 2 || Q > 4 || H < 16 || (int64_t)Q * H > 128) return NVFP4MLA_ERR_INVALID_ARG;
  if (member_masks == nullptr) return NVFP4MLA_ERR_INVALID_ARG;
  if (pointer_kind(member_masks) != kPtrDevice) return NVFP4MLA_ERR_INVALID_ARG;
  FoldArgs fold{member_masks, Q, H};
  return decode_impl(q, kv_cache, num_pages, page_table, max_pages_per_seq, shared_indices, seq_lens, B, 1, Q * H,
                     topk, softmax_scale, out, lse, workspace, workspace_bytes, dev_status, flags, stream, 0, &fold);
}

int sparse_mla_decode_fp8_token(const void* q, const void* kv_cache_tok, int64_t num_pages, const int32_t* page_table,
                                int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens,
                                int B, int Q, int H, int topk, float softmax_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return decode_impl(q, kv_cache_tok, num_pages, page_table, max_pages_per_seq, topk_indices, seq_lens, B, Q, H,
                     topk, softmax_scale, out, lse, workspace, workspace_bytes, dev_status, 0u, stream, 2);
}

// Shared checks of the bf16-row packs (mla_kv_pack's rules); row_bytes of the destination format.
static int check_pack_args(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                           const int64_t* slot_mapping, int64_t num_tokens, const void* cache, int64_t num_pages,
                           const int32_t* dev_status, int row_bytes) {
  if (num_tokens < 0 || num_pages < 1) return NVFP4MLA_ERR_INVALID_ARG;
  if (latent == nullptr || rope == nullptr || slot_mapping == nullptr || cache == nullptr)
    return NVFP4MLA_ERR_INVALID_ARG;
  if (latent_row_stride < kLatent || rope_row_stride < kRope) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages > (INT64_MAX / (kPageTokens * (int64_t)row_bytes))) return NVFP4MLA_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || (latent_row_stride % 8) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(rope, 4) || (rope_row_stride % 2) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(cache, 16) || !aligned(slot_mapping, 8)) return NVFP4MLA_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return NVFP4MLA_ERR_ALIGNMENT;
  if (pointer_kind(latent) != kPtrDevice || pointer_kind(rope) != kPtrDevice ||
      pointer_kind(slot_mapping) != kPtrDevice || pointer_kind(cache) != kPtrDevice ||
      (dev_status != nullptr && pointer_kind(dev_status) != kPtrDevice))
    return NVFP4MLA_ERR_INVALID_ARG;
  return NVFP4MLA_OK;
}

int fp8_token_kv_pack(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                      const int64_t* slot_mapping, int64_t num_tokens, void* kv_cache_tok, int64_t num_pages,
                      int32_t* dev_status, void* stream) {
  if (num_tokens == 0 && num_pages >= 1) return NVFP4MLA_OK;
  const int rc = check_pack_args(latent, latent_row_stride, rope, rope_row_stride, slot_mapping, num_tokens,
                                 kv_cache_tok, num_pages, dev_status, kTokRowBytes);
  if (rc != NVFP4MLA_OK) return rc;
  const cudaError_t err = launch_token_pack(static_cast<const uint16_t*>(latent), latent_row_stride,
                                            static_cast<const uint16_t*>(rope), rope_row_stride, slot_mapping,
                                            num_tokens, static_cast<uint8_t*>(kv_cache_tok), num_pages, dev_status,
                                            static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? NVFP4MLA_OK : NVFP4MLA_ERR_CUDA;
}

int fp8_kv_pack(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                const int64_t* slot_mapping, int64_t num_tokens, void* kv_cache_fp8, int64_t num_pages,
                int32_t* dev_status, void* stream) {
  if (num_tokens < 0 || num_pages < 1) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return NVFP4MLA_OK;
  if (latent == nullptr || rope == nullptr || slot_mapping == nullptr || kv_cache_fp8 == nullptr)
    return NVFP4MLA_ERR_INVALID_ARG;
  if (latent_row_stride < kLatent || rope_row_stride < kRope) return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages > (INT64_MAX / (kPageTokens * kFp8RowBytes))) return NVFP4MLA_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || (latent_row_stride % 8) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(rope, 4) || (rope_row_stride % 2) != 0) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(kv_cache_fp8, 16) || !aligned(slot_mapping, 8)) return NVFP4MLA_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return NVFP4MLA_ERR_ALIGNMENT;
  if (pointer_kind(latent) != kPtrDevice || pointer_kind(rope) != kPtrDevice ||
      pointer_kind(slot_mapping) != kPtrDevice || pointer_kind(kv_cache_fp8) != kPtrDevice ||
      (dev_status != nullptr && pointer_kind(dev_status) != kPtrDevice))
    return NVFP4MLA_ERR_INVALID_ARG;
  const cudaError_t err = launch_fp8_pack(static_cast<const uint16_t*>(latent), latent_row_stride,
                                          static_cast<const uint16_t*>(rope), rope_row_stride, slot_mapping,
                                          num_tokens, static_cast<uint8_t*>(kv_cache_fp8), num_pages, dev_status,
                                          static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? NVFP4MLA_OK : NVFP4MLA_ERR_CUDA;
}

int nvfp4_stage_fp8(const void* kv_cache, int64_t num_pages, const int32_t* page_table, int64_t max_pages_per_seq,
                    const int32_t* topk_indices, const int32_t* seq_lens, int B, int Q, int topk, void* staged,
                    int32_t* staged_indices, int32_t* staged_page_table, int32_t* staged_seq_lens,
                    int32_t* dev_status, void* stream) {
  if (B < 1 || Q < 1 || Q > 16 || topk < kPageTokens || topk > NVFP4MLA_MAX_TOPK || topk % kPageTokens != 0)
    return NVFP4MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_pages_per_seq < 1 || num_pages > INT32_MAX) return NVFP4MLA_ERR_INVALID_ARG;
  if ((int64_t)B * Q * topk > (int64_t)INT32_MAX) return NVFP4MLA_ERR_UNSUPPORTED;   // staged rows in int32
  if (kv_cache == nullptr || page_table == nullptr || topk_indices == nullptr || seq_lens == nullptr ||
      staged == nullptr || staged_indices == nullptr || staged_page_table == nullptr || staged_seq_lens == nullptr)
    return NVFP4MLA_ERR_INVALID_ARG;
  if (!aligned(kv_cache, 16) || !aligned(staged, 16)) return NVFP4MLA_ERR_ALIGNMENT;
  if (!aligned(page_table, 4) || !aligned(topk_indices, 4) || !aligned(seq_lens, 4) || !aligned(staged_indices, 4) ||
      !aligned(staged_page_table, 4) || !aligned(staged_seq_lens, 4))
    return NVFP4MLA_ERR_ALIGNMENT;
  if (dev_status != nullptr && !aligned(dev_status, 4)) return NVFP4MLA_ERR_ALIGNMENT;
  const void* ptrs[8] = {kv_cache, page_table, topk_indices, seq_lens, staged, staged_indices, staged_page_table,
                         staged_seq_lens};
  for (const void* ptr : ptrs)
    if (pointer_kind(ptr) != kPtrDevice) return NVFP4MLA_ERR_INVALID_ARG;
  if (dev_status != nullptr && pointer_kind(dev_status) != kPtrDevice) return NVFP4MLA_ERR_INVALID_ARG;
  const cudaError_t err =
      launch_stage(static_cast<const uint8_t*>(kv_cache), num_pages, page_table, max_pages_per_seq, topk_indices,
                   seq_lens, B, Q, topk, static_cast<uint8_t*>(staged), staged_indices, staged_page_table,
                   staged_seq_lens, dev_status, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? NVFP4MLA_OK : NVFP4MLA_ERR_CUDA;
}

}  // extern "C"
