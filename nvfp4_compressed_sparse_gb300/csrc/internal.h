// Internal declarations shared by the host API and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4mla {

constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kQK = 576;
constexpr int kRowBytes = 352;
constexpr int kFp8RowBytes = 576;   // FP8 comparison rows: 512 latent + 64 rope E4M3 bytes
constexpr int kTokRowBytes = 672;   // per-token FP8 rows: 512 E4M3 latent / scale, 64 bf16 rope / scale, fp32 scale, pad
constexpr int kTokRopeOff = 512;
constexpr int kTokScaleOff = 640;
constexpr int kPageTokens = 64;
constexpr int kScaleOff = 256;
constexpr int kRopeOff = 288;

constexpr int kTileTokens = 128;      // tokens per decode tile (UMMA M)
constexpr int kHeadsPerCta = 32;      // heads handled by one decode CTA (UMMA N <= 32)
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // bounded in-kernel waits: 2 s

// Work split of the decode kernel. Stream-K (cluster == 0): the tiles of all (unit, head-group)
// pairs form one sequence, cut into `ctas` contiguous ranges; the merge grid combines the partials.
// Cluster (cluster == G >= 1): G CTAs (one thread-block cluster) per unit, each a contiguous share
// of the unit's tiles, combined on chip through distributed shared memory.
struct DecodeSchedule {
  int64_t units;           // B * Q * head_groups
  int tiles_per_unit;      // ceil(topk / 128)
  int64_t total_tiles;     // units * tiles_per_unit
  int ctas;                // grid size
  int64_t partial_slots;   // stream-K: ctas + units - 1
  int cluster;             // 0 = stream-K, else CTAs per unit
  int pair;                // 1 = stream-K over pairs: ctas ranges, each run by a 2-CTA cluster (one K half per CTA)
};

// kClusterNone: stream-K split only; kClusterDefault: the policy without flags (the split, measured
// faster); kClusterBalanced: the cluster schedule wherever it is as balanced as the split;
// kClusterAny: whenever one wave of clusters fits. kPairSplit: stream-K over SMs / 2 ranges, each run
// by a 2-CTA cluster whose CTAs hold one half of the 576-wide contraction each.
enum ClusterPolicy { kClusterNone, kClusterDefault, kClusterBalanced, kClusterAny, kPairSplit };
DecodeSchedule make_schedule(int B, int Q, int H, int topk, int num_sms, int max_ctas, ClusterPolicy policy);
size_t workspace_bytes_for(const DecodeSchedule& s, int H);

struct DecodeParams {
  CUtensorMap cache_map;      // 2-D view of the cache: [num_pages*64 rows, row bytes / 4 x uint32], one-row box
  const uint16_t* q;          // bf16 [B, Q, H, 576]
  const uint8_t* cache;       // [num_pages, 64, 352] (FP8 rows: [num_pages, 64, 576])
  int64_t num_pages;
  const int32_t* page_table;  // [B, max_pages]
  int64_t max_pages;
  const int32_t* idx;         // [B, Q, topk] index lists
  const int32_t* seq_lens;    // [B]
  int B, Q, H, topk;
  int heads_per_cta;          // 16 or 32
  int head_groups;            // H / heads_per_cta
  float scale_log2;           // softmax_scale * log2(e)
  uint16_t* out;              // bf16 [B, Q, H, 512]
  float* lse;                 // [B, Q, H]
  float* part_o;              // [slots, heads_per_cta, 512]
  float* part_ml;             // [slots, heads_per_cta, 2]  (running max in log2 units, sum)
  uint8_t* q16;               // [units, 9 * heads_per_cta * 128]: FP16 q image in UMMA B layout
  float* qscale;              // [units]: softmax_scale * log2(e) * 2^-e for the unit's q scaling
  uint64_t* part_flag;        // [slots]: tag of the call whose partial the slot holds (stream-K)
  uint64_t tag;               // this call's tag (unique per call in the process)
  int merge_poll;             // 1 = the merge polls part_flag (results in host memory), else waits for the grid
  int32_t* status;            // optional
  int64_t units, total_tiles;
  int tiles_per_unit, ctas;
  int cluster;                // 0 = stream-K split, else CTAs per unit (one cluster per unit)
  int pair;                   // 1 = the split run by 2-CTA clusters: ctas = ranges (pairs), 2 * ctas CTAs
  uint32_t withhold;          // testing aid: 1 = the producers never publish tile 1's row table
  // Folded queries (sparse_mla_decode_shared): the kernel runs Q = 1 with H = fold_q * fold_h heads, the
  // fold_q query tokens of a request sharing one index list; fold_member[b * topk + e] bit j says whether
  // entry e belongs to query token j. fold_q = 1: no fold.
  const uint8_t* fold_member;
  int fold_q, fold_h;
  int row_fmt;                // 0 = 352-byte NVFP4 rows, 1 = 576-byte FP8 rows, 2 = 672-byte per-token FP8 rows
                              // (1 and 2: split schedule only)
};

cudaError_t launch_pack(const uint16_t* latent, int64_t lstride, const uint16_t* rope, int64_t rstride,
                        const int64_t* slots, int64_t n, uint8_t* cache, int64_t num_pages, int32_t* status,
                        cudaStream_t stream);
cudaError_t launch_fp8_pack(const uint16_t* latent, int64_t lstride, const uint16_t* rope, int64_t rstride,
                            const int64_t* slots, int64_t n, uint8_t* cache, int64_t num_pages, int32_t* status,
                            cudaStream_t stream);
cudaError_t launch_token_pack(const uint16_t* latent, int64_t lstride, const uint16_t* rope, int64_t rstride,
                              const int64_t* slots, int64_t n, uint8_t* cache, int64_t num_pages, int32_t* status,
                              cudaStream_t stream);
cudaError_t launch_stage(const uint8_t* cache, int64_t num_pages, const int32_t* page_table, int64_t max_pages,
                         const int32_t* idx, const int32_t* seq_lens, int B, int Q, int K, uint8_t* staged,
                         int32_t* staged_idx, int32_t* staged_pt, int32_t* staged_sl, int32_t* status,
                         cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
int max_active_clusters(int heads_per_cta, int cluster);   // clusters of the decode grid that fit at once
cudaError_t launch_decode_pair(const DecodeParams& p, cudaStream_t stream);   // the pair grid alone
int max_active_pairs(int heads_per_cta);                    // pairs of the pair grid that fit at once
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream);

cudaError_t launch_topk(const float* logits, int64_t stride, const int32_t* seq_lens, int B, int Q, int K,
                        int32_t* out, cudaStream_t stream);

int device_sm_count();
// Workspace bytes sparse_mla_decode needs for these sizes and flags on the current device (same
// checks and return codes as the call).
int decode_workspace_need(int B, int Q, int H, int topk, uint32_t flags, size_t* need);

}  // namespace nvfp4mla
