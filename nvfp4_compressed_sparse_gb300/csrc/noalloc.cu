// sparse_mla_decode_noalloc: the sparse MLA decode step for callers that cannot
// allocate device memory, using a fixed scratch area built into the library.
//
// Who needs this: code that runs where no allocation may happen and no
// scratch argument can be threaded through -- for example an operator called
// from inside a serving engine that has already reserved (or pinned down) all
// device memory for its own pool, a plugin whose enqueue signature has no
// workspace argument, or a latency-critical path that must never call the CUDA
// allocator. The regular sparse_mla_decode needs a caller-provided workspace;
// this variant takes its scratch from kScratchBytes of device memory that the
// library reserves statically on every GPU where it is loaded (held until the
// process exits).
//
// Rules (also stated in include/nvfp4mla.h):
//  * The first call on a device looks up the scratch address on that device
//    (cudaGetSymbolAddress, with the device current). Make that first call
//    before any stream capture begins.
//  * Every call on a device shares the same scratch. Calls whose kernels
//    overlap on the GPU (different streams without ordering) race and may
//    return wrong results; order them on one stream or with events.
//  * Nothing in the scratch has to start at zero: every byte the kernels read
//    was written earlier in the same call.
//  * Sizes whose scratch need exceeds kScratchBytes are rejected with
//    NVFP4MLA_ERR_WORKSPACE before anything is enqueued.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4mla.h"
#include "internal.h"

namespace nvfp4mla {
namespace {

constexpr size_t kScratchBytes = NVFP4MLA_NOALLOC_SCRATCH_BYTES;   // 32 MiB
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace nvfp4mla

extern "C" int sparse_mla_decode_noalloc(const void* q, const void* kv_cache, int64_t num_pages,
                                         const int32_t* page_table, int64_t max_pages_per_seq,
                                         const int32_t* topk_indices, const int32_t* seq_lens, int B, int Q, int H,
                                         int topk, float softmax_scale, void* out, float* lse, int32_t* dev_status,
                                         uint32_t flags, void* stream) {
  using namespace nvfp4mla;
  // The scratch this call's own schedule needs (the flags can change the grid), with the same
  // size checks and return codes as sparse_mla_decode.
  size_t need = 0;
  const int rc = decode_workspace_need(B, Q, H, topk, flags, &need);
  if (rc != NVFP4MLA_OK) return rc;
  if (need > kScratchBytes) return NVFP4MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return NVFP4MLA_ERR_CUDA;
  return sparse_mla_decode(q, kv_cache, num_pages, page_table, max_pages_per_seq, topk_indices, seq_lens, B, Q, H,
                           topk, softmax_scale, out, lse, scratch, kScratchBytes, dev_status, flags, stream);
}
