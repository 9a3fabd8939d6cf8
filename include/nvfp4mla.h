/*
 * nvfp4mla: NVFP4-compressed paged MLA cache write and sparse MLA decode on
 * GB300 (sm_103a). C ABI; plain pointers and sizes only.
 *
 * The method (sources are named per call below):
 *   "Prime Inference: fast, reliable serving for frontier open models"
 *   (translated launch post), section "Decode: NVFP4 KV compression";
 *   "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem",
 *   sections "Four bits per latent value: where 352 comes from" and "A kernel
 *   that reads four bits directly"; the "TokenSpeed" engine walkthrough,
 *   section 8 "MLA KV layout" and its MLA decode benchmark example.
 *
 * Common rules for every call:
 *   - All pointers except dev_status may be NULL only where stated. Data
 *     pointers are DEVICE pointers of the current CUDA device, except where a
 *     call states that page-locked host memory is accepted.
 *   - The caller owns every buffer. The library never allocates, never frees
 *     and never synchronises; all work is enqueued on `stream` (a
 *     cudaStream_t; NULL = legacy default stream) and the call returns before
 *     the work finishes.
 *   - Problems the host can see (bad sizes, NULL pointers, misalignment, a
 *     workspace that is too small) return a non-zero status before anything
 *     is enqueued. A failed launch returns NVFP4MLA_ERR_CUDA.
 *   - Problems in the data (bad indices, bad page-table entries, bad slots)
 *     never fault: the entry is skipped and counted in dev_status.
 *   - The library keeps no state between calls and may be called from
 *     several host threads at once (on different streams or the same one).
 */
#ifndef NVFP4MLA_H_
#define NVFP4MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
enum {
  NVFP4MLA_OK = 0,
  NVFP4MLA_ERR_INVALID_ARG = 1, /* NULL pointer, negative or unsupported size       */
  NVFP4MLA_ERR_ALIGNMENT = 2,   /* a pointer or stride breaks the alignment rules   */
  NVFP4MLA_ERR_UNSUPPORTED = 3, /* valid request this build does not handle         */
  NVFP4MLA_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required          */
  NVFP4MLA_ERR_CUDA = 5         /* a CUDA call or kernel launch failed              */
};

/* Row format constants (bytes / values). */
#define NVFP4MLA_LATENT_DIM 512   /* latent values per row                        */
#define NVFP4MLA_ROPE_DIM 64      /* rope values per row                          */
#define NVFP4MLA_QK_DIM 576       /* 512 + 64: width of an absorbed query         */
#define NVFP4MLA_ROW_BYTES 352    /* 256 nibble bytes + 32 scale bytes + 64 rope  */
#define NVFP4MLA_PAGE_TOKENS 64   /* tokens per cache page                        */
#define NVFP4MLA_MAX_TOPK 8192    /* largest index list per query                 */

/* Words of the optional device status array (int32[NVFP4MLA_STATUS_WORDS]).
 * The library only ever adds to them (atomically); the caller zeroes them. */
#define NVFP4MLA_STAT_BAD_INDEX 0 /* index entries other than -1 left out: < -1,
                                     >= seq_len, or past the causal position    */
#define NVFP4MLA_STAT_BAD_PAGE 1  /* entries left out because idx/64 is not a
                                     page-table column or the entry is not a
                                     page of the cache                          */
#define NVFP4MLA_STAT_TIMEOUT 2   /* bounded in-kernel waits that gave up; the
                                     outputs of that call are then undefined    */
#define NVFP4MLA_STAT_BAD_SLOT 3  /* pack slots other than -1 outside the cache */
#define NVFP4MLA_STATUS_WORDS 4

/*
 * mla_kv_pack: write bf16 latent + rope rows into the paged NVFP4 cache.
 *
 * Source: "Prime Inference" (translated), "Making room for low-latency
 * decode": the 512-value latent is stored as 4-bit values with one FP8 scale
 * per 16 values and the 64-value rope part as FP8, 352 bytes per row; the
 * byte split is the table of "Four bits per latent value: where 352 comes
 * from". The call shape follows the cache-write call of the TokenSpeed
 * walkthrough, section 8 (location list + latent + rope).
 *
 * Per row: for each block k of 16 latent values, s_k = E4M3(amax_k / 6)
 * (nearest-even, saturating at 448); each value is coded as e2m1(x / s_k)
 * (nearest-even, saturating at 6, sign kept; all magnitudes 0 when s_k = 0).
 * Row bytes: [0,256) nibbles, element 2i in the low nibble of byte i;
 * [256,288) the 32 scales; [288,352) E4M3(rope[d]).
 * Non-finite inputs (the pages are silent; this library's rule): a NaN
 * latent value takes no part in its block's amax and is stored with
 * magnitude 0 (sign kept); an infinity saturates its block scale to 448 and
 * is stored as +-6; a NaN rope value is stored as E4M3 NaN (0x7F or 0xFF,
 * sign kept), an infinite one as +-448.
 *
 *   latent            bf16 [num_tokens, 512], row stride latent_row_stride
 *                     ELEMENTS; base 16-byte aligned, stride a multiple of 8
 *   rope              bf16 [num_tokens, 64], row stride rope_row_stride
 *                     elements; base 4-byte aligned, stride a multiple of 2
 *   slot_mapping      int64 [num_tokens]; token t goes to page slot/64, row
 *                     slot%64; -1 = skip the token; other out-of-range slots
 *                     are skipped and counted (NVFP4MLA_STAT_BAD_SLOT)
 *   num_tokens        >= 0 (0 enqueues nothing and returns OK)
 *   kv_cache          uint8 [num_pages, 64, 352], 16-byte aligned; rows not
 *                     named by a slot are left untouched
 *   num_pages         >= 1
 *   dev_status        optional int32[NVFP4MLA_STATUS_WORDS] (may be NULL)
 *   stream            cudaStream_t
 * All pointers must be device memory of the current device: each is checked
 * with cudaPointerGetAttributes first, and host memory (pageable or
 * page-locked), another device's memory or an unknown pointer returns
 * NVFP4MLA_ERR_INVALID_ARG with nothing enqueued.
 * Two tokens mapped to the same slot race; the caller must not do that.
 */
int mla_kv_pack(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                const int64_t* slot_mapping, int64_t num_tokens, void* kv_cache, int64_t num_pages,
                int32_t* dev_status, void* stream);

/*
 * sparse_mla_decode_workspace_size: bytes of device workspace that
 * sparse_mla_decode needs for these sizes on a GPU with num_sms SMs
 * (num_sms <= 0: ask the current device). Returns 0 for invalid sizes.
 */
size_t sparse_mla_decode_workspace_size(int B, int Q, int H, int topk, int num_sms);

/*
 * sparse_mla_decode: one MLA decode step over the paged NVFP4 cache, each
 * query attending only to its indexer-selected positions.
 *
 * Source: "Prime Inference" (translated), "Native NVFP4 sparse MLA decode
 * kernel": load the selected compressed rows, unpack them on chip, score,
 * softmax and blend with 16-bit operands and FP32 accumulation; -1 entries are
 * unused and are not read. "Serving GLM-5.3 ...", "Prefill topology": one
 * 512 + 64 row per token shared by every head. TokenSpeed MLA decode
 * example: page size 64, softmax scale 1/sqrt(192).
 *
 * For query (b, j) and head h, with C_t the dequantised row of position t
 * (latent e2m1 * E4M3 scale, rope E4M3) and T the multiset of usable entries
 * of topk_indices[b, j, :]:
 *   z_t = softmax_scale * <q[b,j,h,:], C_t>           (576-wide)
 *   out[b,j,h,:] = sum_t exp(z_t - m) C_t[0:512] / sum_t exp(z_t - m)
 *   lse[b,j,h]   = m + ln(sum_t exp(z_t - m)),  m = max_t z_t
 * An entry idx is usable iff 0 <= idx < seq_lens[b], idx <= seq_lens[b]-Q+j
 * (causal within the Q new tokens), idx/64 < max_pages_per_seq and
 * 0 <= page_table[b, idx/64] < num_pages. Entries are counted as often as
 * listed. A query with no usable entry gets out = 0 and lse = -inf.
 *
 * Host buffers: q, page_table, topk_indices, seq_lens, out and lse may each be
 * page-locked host memory mapped for the device at the same address
 * (cudaMallocHost / cudaHostAlloc, or cudaHostRegister'd; on GB300 the GPU
 * reaches it over NVLink-C2C). The kernels then read those inputs from, and
 * write the results to, host memory themselves, in stream order, with results
 * identical to device buffers; no separate copy is needed. kv_cache, workspace
 * and dev_status must be device memory. Every pointer is checked with
 * cudaPointerGetAttributes before anything is enqueued: pageable host memory,
 * another device's memory or an unknown pointer returns
 * NVFP4MLA_ERR_INVALID_ARG.
 *
 *   q                 bf16 [B, Q, H, 576] contiguous, 16-byte aligned
 *   kv_cache          uint8 [num_pages, 64, 352], 16-byte aligned
 *   page_table        int32 [B, max_pages_per_seq] contiguous
 *   topk_indices      int32 [B, Q, topk] contiguous; logical positions, -1 =
 *                     unused
 *   seq_lens          int32 [B]; cached tokens of request b including its Q
 *                     new tokens
 *   B, Q, H, topk     B >= 1, 1 <= Q <= 16, H in {16, 32, 64, 128},
 *                     1 <= topk <= NVFP4MLA_MAX_TOPK
 *   softmax_scale     > 0 (typically 1/sqrt(192))
 *   out               bf16 [B, Q, H, 512] contiguous, 16-byte aligned
 *   lse               fp32 [B, Q, H] (natural log)
 *   workspace         device scratch of at least
 *                     sparse_mla_decode_workspace_size(B, Q, H, topk, 0)
 *                     bytes, 256-byte aligned; contents need no
 *                     initialisation and are clobbered
 *   dev_status        optional int32[NVFP4MLA_STATUS_WORDS] (may be NULL)
 *   flags             0 (the split schedule, see sparse_mla_decode_plan), or
 *                     NVFP4MLA_FLAG_MAX_CTAS(n) to cap the number of decode
 *                     CTAs at n (testing aid; 0 = no cap; a cap also selects
 *                     the split schedule), optionally or-ed with
 *                     NVFP4MLA_FLAG_SPLIT (always the split schedule) or
 *                     NVFP4MLA_FLAG_CLUSTER (also take the cluster schedule
 *                     wherever it is as balanced as the split one) and, with
 *                     it, NVFP4MLA_FLAG_CLUSTER_ANY (tuning aid: take the
 *                     cluster schedule whenever one wave of clusters fits),
 *                     or NVFP4MLA_FLAG_PAIR (the pair schedule, see
 *                     sparse_mla_decode_plan; results in device memory
 *                     only, else the split schedule is used), optionally
 *                     or-ed with NVFP4MLA_FLAG_TEST_TIMEOUT (testing aid: the
 *                     decode grid withholds one internal signal, so its
 *                     bounded waits expire after about 2 s; the grid then
 *                     counts the timeout in dev_status[NVFP4MLA_STAT_TIMEOUT],
 *                     drains its copies and returns; out and lse are
 *                     undefined)
 *   stream            cudaStream_t
 * Calls that share a workspace must be ordered on one stream.
 */
#define NVFP4MLA_FLAG_MAX_CTAS(n) ((uint32_t)(n) & 0xFFFFu)
#define NVFP4MLA_FLAG_TEST_TIMEOUT (1u << 31)
#define NVFP4MLA_FLAG_CLUSTER (1u << 30)
#define NVFP4MLA_FLAG_CLUSTER_ANY (1u << 29)
#define NVFP4MLA_FLAG_SPLIT (1u << 28)
#define NVFP4MLA_FLAG_PAIR (1u << 27)
int sparse_mla_decode(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* page_table,
                      int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens, int B,
                      int Q, int H, int topk, float softmax_scale, void* out, float* lse, void* workspace,
                      size_t workspace_bytes, int32_t* dev_status, uint32_t flags, void* stream);

/*
 * sparse_mla_decode_plan: the decode grid that sparse_mla_decode launches for
 * these sizes and flags on the current device. (The pages give no such call;
 * it reports this library's schedule.)
 *
 * Source: "Prime Inference" (translated), "Native NVFP4 sparse MLA decode
 * kernel": the selected rows of one query token are split over a cluster of
 * SMs whose partial results are merged on chip, the cluster size adapted to
 * the batch. Two schedules:
 *   - cluster (*cluster = G >= 1): G CTAs (one thread-block cluster, G <= 8)
 *     per (query, head group); each takes a contiguous share of its selected
 *     rows, q is converted in the decode grid and the partials are merged
 *     through distributed shared memory inside the same grid: one launch.
 *   - split (*cluster = 0): the 128-row tiles of all queries form one
 *     sequence cut into *ctas contiguous ranges (one CTA per SM); a q-prep
 *     grid runs before it and a merge grid combines the partials.
 * Without flags the split schedule is used: on GB300 it measured faster at
 * every size tried (64 queries: 50.0 vs 52.8 us with 2-CTA clusters; 128
 * queries, an earlier build: 93.9 vs 96.9 us with 1-CTA clusters; 1 and 4
 * queries: ~6 us faster than 8-CTA clusters). NVFP4MLA_FLAG_CLUSTER takes the cluster schedule when
 * one wave of clusters fits and no CTA runs more 128-row tiles than under the
 * split schedule; NVFP4MLA_FLAG_CLUSTER_ANY whenever one wave fits.
 * A third, opt-in schedule (NVFP4MLA_FLAG_PAIR, *cluster = -2) runs the
 * split schedule's ranges on 2-CTA clusters (*ctas = 2 x SMs / 2): CTA h of a
 * pair holds half h of the 576-wide contraction (latent dims 256h..256h+255
 * and rope dims 32h..32h+31), the two exchange their partial scores every
 * 128-row tile through distributed shared memory, and the freed on-chip
 * memory double-buffers K and S and lets PV read V once for both parts of P.
 * Measured on GB300 (headline rows, L2 flushed): 67.7 vs 50.0 us for 64
 * queries, 33.6 vs 29.6 us for 16, 23.4 vs 21.5 us for 4, 21.7 vs 21.0 for 1; each
 * SM then runs the softmax of twice as many tile visits, and the exchange
 * adds a dependency between the CTAs every tile.
 *   B, Q, H, topk     as for sparse_mla_decode
 *   flags             as for sparse_mla_decode
 *   ctas, cluster     host int pointers (either may be NULL): the grid size
 *                     and G (0 = split schedule, -2 = pair schedule)
 * Returns NVFP4MLA_OK, NVFP4MLA_ERR_INVALID_ARG for invalid sizes, or
 * NVFP4MLA_ERR_CUDA when the device cannot be queried.
 */
int sparse_mla_decode_plan(int B, int Q, int H, int topk, uint32_t flags, int* ctas, int* cluster);

/*
 * sparse_mla_decode_noalloc: sparse_mla_decode for callers that cannot
 * allocate device memory. (The pages describe no such call; this is a
 * deployment convenience of this library.)
 *
 * Some callers cannot allocate or pass a scratch buffer: an operator running
 * inside a serving engine that has reserved all device memory for its own
 * pool, a plugin whose enqueue signature has no workspace argument, or a path
 * that must never enter the CUDA allocator. This call computes exactly what
 * sparse_mla_decode computes, with the same arguments minus the workspace; its
 * scratch is a fixed NVFP4MLA_NOALLOC_SCRATCH_BYTES region of device memory
 * that the library reserves statically on every GPU where it is loaded (held
 * until the process exits). It allocates nothing.
 *   - The first call on a device looks up that region's address on the
 *     current device; make the first call before any stream capture starts.
 *   - All calls on a device share the region: calls whose work overlaps on the
 *     GPU race. Order them on one stream (or with events).
 *   - The region needs no initialisation; each call writes what it reads.
 *   - Returns NVFP4MLA_ERR_WORKSPACE, before enqueuing anything, when the call
 *     (these sizes and flags, on the current device) needs more scratch than
 *     the region holds; otherwise as sparse_mla_decode (same size checks and
 *     return codes).
 */
#define NVFP4MLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int sparse_mla_decode_noalloc(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* page_table,
                              int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens, int B,
                              int Q, int H, int topk, float softmax_scale, void* out, float* lse, int32_t* dev_status,
                              uint32_t flags, void* stream);

/*
 * indexer_topk: the index lists sparse_mla_decode reads, from the indexer's
 * logits: for each query token, the top-k positions of its causal range.
 *
 * Source: "Prime Inference: serving GLM-5.3 to agents is a KV-cache
 * problem", section "Decode: TP4, and the copies it keeps" (the indexer keeps
 * the top-2,048 positions of a query); "Prime Inference" (translated), "Native
 * NVFP4 sparse MLA decode kernel" (unused list entries are -1). The pages do
 * not define the indexer's logits; they are this call's input.
 *
 * For query j of request b, the candidate positions are 0 .. seq_lens[b]-Q+j
 * (the decode's causal rule), capped at logits_row_stride. The topk largest
 * logits are selected; logits compare as floats with NaN below every number
 * and -0.0 below +0.0, and among equal logits the smaller position is taken
 * first. topk_indices[b, j, :] lists the selected positions in increasing
 * order; when the range is shorter than topk, all of it is listed and the
 * rest is -1. The result is exact (no approximation, deterministic).
 *
 *   logits            fp32 [B, Q, logits_row_stride] device memory; row (b, j)
 *                     starts at logits + (b*Q + j) * logits_row_stride;
 *                     16-byte aligned, stride a multiple of 4, 1 <= stride
 *                     <= INT32_MAX
 *   seq_lens          int32 [B] device memory: cached tokens of request b,
 *                     including its Q new tokens
 *   B, Q, topk        B >= 1, 1 <= Q <= 16, 1 <= topk <= NVFP4MLA_MAX_TOPK
 *   topk_indices      int32 [B, Q, topk] device memory (output)
 *   stream            cudaStream_t
 * Returns NVFP4MLA_OK, NVFP4MLA_ERR_INVALID_ARG (bad sizes, NULL, memory that
 * is not device memory of the current device), NVFP4MLA_ERR_ALIGNMENT or
 * NVFP4MLA_ERR_CUDA; nothing is enqueued on an error.
 */
int indexer_topk(const float* logits, int64_t logits_row_stride, const int32_t* seq_lens, int B, int Q, int topk,
                 int32_t* topk_indices, void* stream);

/*
 * sparse_mla_decode_shared: one decode step for the Q query tokens of each
 * request (speculative verify: draft tokens) folded into one pass over a
 * shared index list ("TokenSpeed" walkthrough, MLA decode section: fold_sq
 * folds the query-token axis into the head axis). Each cached row the request
 * selects is gathered and unpacked once and scored for the Q * H (query, head)
 * columns together, instead of once per query token.
 *   shared_indices    int32 [B, topk]: the request's positions (any order, -1
 *                     unused), the union of its query tokens' lists
 *   member_masks      uint8 [B, topk] device memory: bit j set when entry e
 *                     belongs to query token j's list
 *   Q, H              2 <= Q <= 4, H >= 16, Q * H in {32, 64, 128}: the
 *                     kernel treats the step as one query of Q * H heads, in
 *                     head groups of 32 (so 32 / H query tokens share a pass)
 *   everything else   as sparse_mla_decode (q [B, Q, H, 576], out
 *                     [B, Q, H, 512], lse [B, Q, H]; workspace
 *                     sparse_mla_decode_workspace_size(B, 1, Q * H, topk, 0)),
 *                     except that the call always takes the split schedule
 *                     (cluster flags are ignored) and out and lse must be
 *                     device memory (else NVFP4MLA_ERR_UNSUPPORTED)
 * Query token j attends exactly to the entries with bit j set that are usable
 * under sparse_mla_decode's rule for query j (0 <= idx < seq_len,
 * idx <= seq_len - Q + j, a valid page): the result equals sparse_mla_decode
 * on per-query lists that hold those entries. Entries invalid for every query
 * are counted in dev_status as sparse_mla_decode counts them.
 * Returns as sparse_mla_decode; NVFP4MLA_ERR_INVALID_ARG for unsupported Q, H.
 */
int sparse_mla_decode_shared(const void* q, const void* kv_cache, int64_t num_pages, const int32_t* page_table,
                             int64_t max_pages_per_seq, const int32_t* shared_indices, const uint8_t* member_masks,
                             const int32_t* seq_lens, int B, int Q, int H, int topk, float softmax_scale, void* out,
                             float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status, uint32_t flags,
                             void* stream);

/*
 * FP8 comparison paths. The pages compare the native NVFP4 decode with (i) a
 * staged path, where a gather kernel unpacks each selected 352-byte NVFP4 row
 * into a 576-byte FP8 copy in GPU memory and an FP8 attention kernel reads the
 * copy (352 + 576 + 576 = 1,504 bytes per selected row), and (ii) an FP8
 * attention kernel over a cache of 576-byte FP8 rows ("Prime Inference:
 * serving GLM-5.3 to agents is a KV-cache problem", section "A kernel that
 * reads four bits directly"; "Prime Inference" (translated), "Native NVFP4
 * sparse MLA decode kernel"). These entry points build both on GB300 with the
 * same decode kernel, so the three paths differ only in the bytes they move.
 *
 * FP8 row (576 bytes): byte d < 512 is E4M3 of latent value d, byte 512 + r is
 * E4M3 of rope value r; no scale. E4M3 rounding: nearest, ties to even,
 * saturating at +-448; NaN becomes 0x7F with its sign bit.
 */

/*
 * fp8_kv_pack: bf16 latent + rope rows -> 576-byte FP8 rows of a paged cache
 * uint8 [num_pages, 64, 576] (device memory). Arguments, checks, slot rules and
 * dev_status counting are those of mla_kv_pack.
 */
int fp8_kv_pack(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                const int64_t* slot_mapping, int64_t num_tokens, void* kv_cache_fp8, int64_t num_pages,
                int32_t* dev_status, void* stream);

/*
 * nvfp4_stage_fp8: the staging kernel of the staged path, for one decode
 * step over an NVFP4 cache. For query (b, j) and list entry i it applies the
 * decode's entry rule (see sparse_mla_decode); a usable entry's row is copied
 * to staged row (b*Q + j)*topk + i as an FP8 row (latent value e2m1(code) x
 * E4M3(scale), exact, rounded once to E4M3; a block with a NaN scale byte
 * becomes 0x7F; rope bytes copied) and staged_indices[b*Q + j, i] = i;
 * unusable entries get -1 and their staged rows are not written. It also
 * writes staged_page_table[u, p] = u*(topk/64) + p and staged_seq_lens[u] =
 * topk, so that sparse_mla_decode_fp8 over the staged rows as B*Q one-query
 * requests (q viewed as [B*Q, 1, H, 576], cache = staged viewed as
 * [B*Q*topk/64, 64, 576], max_pages_per_seq = topk/64) computes the step.
 *   kv_cache ... seq_lens, B, Q   as sparse_mla_decode (device memory)
 *   topk              64 <= topk <= NVFP4MLA_MAX_TOPK, a multiple of 64
 *   staged            uint8 [B*Q*topk, 576] device memory, 16-byte aligned
 *   staged_indices    int32 [B*Q, topk] device memory
 *   staged_page_table int32 [B*Q, topk/64] device memory
 *   staged_seq_lens   int32 [B*Q] device memory
 *   dev_status        optional; counts bad index and bad page entries as
 *                     sparse_mla_decode does
 * Returns NVFP4MLA_OK, NVFP4MLA_ERR_INVALID_ARG, NVFP4MLA_ERR_ALIGNMENT,
 * NVFP4MLA_ERR_UNSUPPORTED (B*Q*topk > INT32_MAX) or NVFP4MLA_ERR_CUDA.
 */
int nvfp4_stage_fp8(const void* kv_cache, int64_t num_pages, const int32_t* page_table, int64_t max_pages_per_seq,
                    const int32_t* topk_indices, const int32_t* seq_lens, int B, int Q, int topk, void* staged,
                    int32_t* staged_indices, int32_t* staged_page_table, int32_t* staged_seq_lens,
                    int32_t* dev_status, void* stream);

/*
 * sparse_mla_decode_fp8: sparse_mla_decode over a cache of 576-byte FP8 rows
 * (uint8 [num_pages, 64, 576], device memory): the same arguments, entry
 * rules, outputs and workspace (sparse_mla_decode_workspace_size), computed
 * by the same kernel with E4M3 -> fp16 conversion in place of the NVFP4
 * unpacking. Always the split schedule; out and lse must be device memory
 * (else NVFP4MLA_ERR_UNSUPPORTED).
 */
int sparse_mla_decode_fp8(const void* q, const void* kv_cache_fp8, int64_t num_pages, const int32_t* page_table,
                          int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens, int B,
                          int Q, int H, int topk, float softmax_scale, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Per-token FP8 comparison path: the per-token FP8 cache of the "TokenSpeed"
 * engine walkthrough (section 8, "MLA KV layout", its per_token_head write
 * path: the latent divided by scale = max(amax, 1e-26) / 448 of the token,
 * stored as E4M3; the rope divided by the same scale, kept in bf16; the scale
 * in fp32). GB300 layout (672 bytes per row): bytes 0..511 the E4M3 codes,
 * 512..639 the 64 bf16 rope values, 640..643 the fp32 scale (little-endian),
 * 644..671 zero. Four rows are a whole number of 128-byte units, so a gather
 * of four rows lands on the 128-byte boundaries the TMA unit requires.
 *
 * fp8_token_kv_pack: bf16 latent + rope rows -> such rows of a paged cache
 * uint8 [num_pages, 64, 672] (device memory); amax, scale and divisions in
 * IEEE fp32, then E4M3 (nearest even, saturating) and bf16 (nearest even).
 * Arguments, checks, slot rules and dev_status counting as mla_kv_pack;
 * inputs must be finite (a NaN or an infinity gives an unspecified row).
 */
int fp8_token_kv_pack(const void* latent, int64_t latent_row_stride, const void* rope, int64_t rope_row_stride,
                      const int64_t* slot_mapping, int64_t num_tokens, void* kv_cache_tok, int64_t num_pages,
                      int32_t* dev_status, void* stream);

/*
 * sparse_mla_decode_fp8_token: sparse_mla_decode over a per-token FP8 cache
 * (uint8 [num_pages, 64, 672], device memory): the same arguments, entry rules,
 * outputs and workspace. The kernel scores q against E4M3 / bf16 values
 * converted to fp16 (the rope exactly for values in fp16's normal range) and
 * applies each row's scale to its score and to its softmax weight. Always the
 * split schedule; out and lse must be device memory (else
 * NVFP4MLA_ERR_UNSUPPORTED).
 */
int sparse_mla_decode_fp8_token(const void* q, const void* kv_cache_tok, int64_t num_pages, const int32_t* page_table,
                                int64_t max_pages_per_seq, const int32_t* topk_indices, const int32_t* seq_lens,
                                int B, int Q, int H, int topk, float softmax_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Human-readable name of a return code (static string, never NULL). */
const char* nvfp4mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MLA_H_ */
