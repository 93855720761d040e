// Indexer scoring + top-K for callers that cannot allocate device memory.
//
// hs_indexer_topk keeps its int64 scores in scratch that hs_pool_init sized and
// allocated. Some callers cannot make that allocation, or any other: an engine
// that hands every free byte of HBM to its KV pool before serving starts (a new
// cudaMalloc then fails or fragments the pool), or code that runs while a stream
// is being captured, where cudaMalloc is not allowed. This entry point runs the
// same kernels with the score scratch in a fixed array inside the library, so
// the call allocates nothing and needs no pool-owned scratch.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its 16 MiB until the process exits. Host code cannot use the
// array's name as a device address (it names a host-side stand-in), so the
// address is taken with cudaGetSymbolAddress once per device, on the first call
// made with that device current, and passed to the kernels.
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "hs_internal.cuh"

using namespace hs;

namespace {

constexpr long long kMaxScores = HS_NOALLOC_MAX_SCORES;   // 2^21 int64 scores = 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int64_t hs_noalloc_scores[kMaxScores];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the static score array on the current device (set-up on first use).
hs_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, hs_noalloc_scores) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return HS_OK;
}

}  // namespace

extern "C" hs_status hs_indexer_topk_noalloc(hs_pool* p, int32_t index_layer, int32_t n, const int32_t* d_req,
                                             const int32_t* d_limit, const int8_t* d_q, const int8_t* d_w,
                                             int32_t* d_topk, hs_stream_t stream) {
  nvtxRangePushA("hs_indexer_topk_noalloc");
  struct Pop {
    ~Pop() { nvtxRangePop(); }
  } pop;
  if (!p || index_layer < 0 || index_layer >= p->d.n_groups || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  if (n == 0) return HS_OK;
  if (!d_req || !d_limit || !d_q || !d_w || !d_topk || (reinterpret_cast<uintptr_t>(d_q) & 15)) return HS_ERR_INVALID;
  if (p->d.idx_fmt != HS_IDX_INT8) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if ((long long)n * p->cfg.max_ctx > kMaxScores) return HS_ERR_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  if (dev != p->device) return HS_ERR_INVALID;
  void* scratch = nullptr;
  hs_status s = scratch_address(dev, &scratch);
  if (s != HS_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int64_t* scores = static_cast<int64_t*>(scratch);
  s = launch_indexer(p, index_layer, n, d_req, d_limit, d_q, d_w, scores, nullptr, st);
  if (s != HS_OK) return s;
  // the cluster selection: it needs no pool-owned scratch
  return launch_select(p, n, scores, p->cfg.max_ctx, d_limit, d_topk, st, false, false);
}
