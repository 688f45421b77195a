// v4a_index_topk_noalloc: the indexer + top-k call for callers that cannot allocate device
// memory and cannot hand the library a workspace either.
//
// Who needs this: a host program that embeds the library inside a framework or a serving
// runtime that owns every byte of device memory (its own arena or pool) and offers a kernel
// library no scratch buffer, or a code path that must not allocate because an allocation
// would synchronise the device or grow a memory budget that has been fixed up front. Such a
// caller still provides the inputs and the output list; the intermediate score rows live
// in a fixed array that is part of the library's device image.
//
// The scratch: kNoallocScoreBytes (8 MiB) in a file-scope __device__ array. Every GPU that
// loads the library holds it until the process exits. A call needs n_q * visible(max_pos)
// fp32 scores; a larger request is refused with V4A_ERR_TOO_LARGE before anything is
// enqueued. The first call on each device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and keeps it for the life of the
// process; make that first call before any stream capture. A device reset
// (cudaDeviceReset) unloads the library's device image, so the kept address is no longer
// valid: do not call this entry point on a device after resetting it. All calls share the one array and it keeps the last call's
// contents: every score the selection reads is written earlier in the same call, so nothing
// has to be cleared, but two calls whose kernels overlap on the GPU (different streams
// without ordering between them) race on the array and give wrong lists.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace v4a {
namespace {

constexpr size_t kNoallocScoreBytes = size_t(8) << 20;
constexpr size_t kNoallocScoreFloats = kNoallocScoreBytes / sizeof(float);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scores[kNoallocScoreFloats];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return V4A_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scores) != cudaSuccess || !p) return V4A_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return V4A_OK;
}

}  // namespace
}  // namespace v4a

using namespace v4a;

extern "C" size_t v4a_index_topk_noalloc_capacity(void) { return kNoallocScoreFloats; }

extern "C" int v4a_index_topk_noalloc(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                                      const int64_t* q_pos, int64_t max_pos, const void* q_idx,
                                      const float* w, const v4a_cache* idx, int32_t k,
                                      int32_t* topk_out, int32_t* dev_err, v4a_stream_t stream) {
  // the same host checks, in the same order, as v4a_index_topk
  IndexParams p{};
  int64_t max_vis = 0;
  int rc = prepare_index(cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, idx, k, topk_out, true,
                         dev_err, &p, &max_vis);
  if (rc || n_q == 0) return rc;
  if ((uint64_t)n_q * (uint64_t)p.row_stride > kNoallocScoreFloats) return V4A_ERR_TOO_LARGE;

  float* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  p.scores = scratch;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = launch_index_scores(p, cfg->dtype, max_vis, st))) return rc;
  return launch_topk(p, max_vis, st);
}
