// Pool state, host-side residency updates, row append, page materialisation and
// the exported C ABI of libhisparse.so.
//
// "vLLM introduces Hybrid HiSparse hybrid sparse offloading for GLM 5.3" (vLLM
// blog Part 1), section "How it works": residency is tracked per page in a
// block table of real blocks and empty placeholders; hot-buffer pages are leased
// from the same pool; completed prefix pages of all sparse-MLA layers are copied
// to host memory in one launch after the forward pass, ordered on the model's
// stream. The big buffers (KV tensors, index caches, pinned host pool) belong to
// the caller; the pool owns only its metadata and scratch, allocated here once.
#include <cstdio>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "hs_select.cuh"

using namespace hs;

namespace {

#define HS_CUDA_TRY(x)                        \
  do {                                        \
    if ((x) != cudaSuccess) return HS_ERR_CUDA; \
  } while (0)

template <typename T>
hs_status dev_alloc(hs_pool* p, T** out, size_t count, int fill_byte) {
  void* ptr = nullptr;
  size_t bytes = count * sizeof(T);
  if (bytes == 0) bytes = 16;
  if (cudaMalloc(&ptr, bytes) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_OOM;
  }
  p->allocations.push_back(ptr);
  if (cudaMemset(ptr, fill_byte, bytes) != cudaSuccess) return HS_ERR_CUDA;
  *out = static_cast<T*>(ptr);
  return HS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---- append: new KV rows (all layers) and index keys (all indexer layers) ----
__global__ void append_kernel(Dev D, int n, const int32_t* __restrict__ req_of, const int32_t* __restrict__ pos_of,
                              const uint8_t* __restrict__ kv_rows, const int8_t* __restrict__ idx_keys) {
  griddep_wait();
  griddep_launch();
  const long long kv_chunks = (long long)n * D.n_layers * ROW_CHUNKS;
  // key record per (token, group): 8 chunks of 16 bytes, plus the fp32 scale (HS_IDX_FP8)
  const bool fp8 = D.idx_fmt == HS_IDX_FP8;
  const int rec = fp8 ? 132 : IDX_DIM;
  const int rec_parts = fp8 ? 9 : 8;
  const long long ix_chunks = (long long)n * D.n_groups * rec_parts;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < kv_chunks + ix_chunks;
       c += (long long)gridDim.x * blockDim.x) {
    if (c < kv_chunks) {
      const int part = (int)(c % ROW_CHUNKS);
      const long long tl = c / ROW_CHUNKS;
      const int layer = (int)(tl % D.n_layers);
      const int t = (int)(tl / D.n_layers);
      const int r = req_of[t], pos = pos_of[t];
      if (r < 0 || r >= D.max_requests || pos < 0 || pos >= D.max_ctx) { set_status(D.status, HS_ERR_BAD_ID); continue; }
      const int pg = D.bt[(size_t)r * D.max_pages + (pos >> 6)];
      if (pg < 0 || pg >= D.num_pages) { set_status(D.status, HS_ERR_BAD_ID); continue; }
      const uint4 v = *reinterpret_cast<const uint4*>(kv_rows + ((size_t)t * D.n_layers + layer) * ROW + part * 16);
      *reinterpret_cast<uint4*>(D.kv[layer] + ((size_t)pg * PAGE + (pos & 63)) * ROW + part * 16) = v;
    } else {
      const long long cc = c - kv_chunks;
      const int part = (int)(cc % rec_parts);
      const long long tg = cc / rec_parts;
      const int g = (int)(tg % D.n_groups);
      const int t = (int)(tg / D.n_groups);
      const int r = req_of[t], pos = pos_of[t];
      if (r < 0 || r >= D.max_requests || pos < 0 || pos >= D.max_ctx) { set_status(D.status, HS_ERR_BAD_ID); continue; }
      const int ip = D.idx_bt[(size_t)r * D.max_pages + (pos >> 6)];
      if (ip < 0 || ip >= D.num_idx_pages) { set_status(D.status, HS_ERR_BAD_ID); continue; }
      const int8_t* src = idx_keys + ((size_t)t * D.n_groups + g) * rec;
      int8_t* page = D.idx[g] + (size_t)ip * D.idx_page_bytes;
      if (part < 8) {   // 128 key bytes (the FP8 record is only 4-byte aligned: copy by words)
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src + part * 16);
        *reinterpret_cast<uint4*>(page + (pos & 63) * IDX_DIM + part * 16) = make_uint4(s32[0], s32[1], s32[2], s32[3]);
      } else {          // the key's fp32 scale, after the page's 64 keys
        *reinterpret_cast<uint32_t*>(page + PAGE * IDX_DIM + (pos & 63) * 4) =
            *reinterpret_cast<const uint32_t*>(src + IDX_DIM);
      }
    }
  }
}

// ---- page materialisation: pool page -> host page, every sparse layer ----
__global__ void offload_kernel(Dev D, int n, const int32_t* __restrict__ pool_pages,
                               const int64_t* __restrict__ host_pages) {
  griddep_wait();
  griddep_launch();
  constexpr int PAGE_CHUNKS = PAGE * ROW / 16;   // 2,624 per page per layer
  const long long total = (long long)n * D.n_layers * PAGE_CHUNKS;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int part = (int)(c % PAGE_CHUNKS);
    const long long il = c / PAGE_CHUNKS;
    const int layer = (int)(il % D.n_layers);
    const int i = (int)(il / D.n_layers);
    const int pg = pool_pages[i];
    const int64_t hp = host_pages[i];
    if (pg < 0 || pg >= D.num_pages || hp < 0 || hp >= D.host_pages) {
      if (part == 0) set_status(D.status, HS_ERR_BAD_ID);
      continue;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(D.kv[layer] + (size_t)pg * PAGE * ROW + part * 16);
    *reinterpret_cast<uint4*>(D.host + ((size_t)hp * D.n_layers + layer) * PAGE * ROW + part * 16) = v;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0)
    atomicAdd(&D.counters[C_D2H], (unsigned long long)n * D.n_layers * PAGE * ROW);
}

__global__ void clear_hot_kernel(Dev D, int r) {
  for (int g = 0; g < D.n_groups; ++g) {
    const size_t rg = (size_t)r * D.n_groups + g;
    for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < D.hot_rows; s += gridDim.x * blockDim.x) {
      D.slot_token[rg * D.hot_rows + s] = -1;
      D.slot_stamp[rg * D.hot_rows + s] = -1;
    }
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < D.max_ctx; t += gridDim.x * blockDim.x)
      D.tok2slot[rg * D.max_ctx + t] = -1;
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < D.hot_pages_max; k += gridDim.x * blockDim.x)
      D.hot_pages[rg * D.hot_pages_max + k] = -1;
    if (blockIdx.x == 0 && threadIdx.x == 0) D.n_hot[rg] = 0;
  }
}

// Host-link probe: n single rows from mapped host memory, 16 B per thread, four
// loads in flight per thread (the resolver's miss-copy pattern).
__global__ void __launch_bounds__(256) link_probe_kernel(const uint8_t* __restrict__ src, long long n_src_rows,
                                                         int row_bytes, const int64_t* __restrict__ rows,
                                                         long long n, uint8_t* __restrict__ dst) {
  const int chunks = row_bytes / 16;
  const long long total = n * chunks;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long c0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; c0 < total; c0 += 4 * stride) {
    uint4 v[4];
    long long at[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long c = c0 + u * stride;
      at[u] = -1;
      if (c >= total) continue;
      const long long i = c / chunks;
      const int part = (int)(c - i * chunks);
      const long long r = rows[i];
      if (r < 0 || r >= n_src_rows) continue;
      v[u] = *reinterpret_cast<const uint4*>(src + (size_t)r * row_bytes + part * 16);
      at[u] = (long long)i * row_bytes + part * 16;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (at[u] >= 0) *reinterpret_cast<uint4*>(dst + at[u]) = v[u];
  }
}

// One NVTX range per ABI call (host side; inert unless a profiler is attached).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
};

// Self-test of the bounded device wait: an mbarrier expecting two arrivals gets one,
// so the wait the hot-path kernels use runs out and records HS_ERR_TIMEOUT.
__global__ void wait_selftest_kernel(Dev D) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 2);
    fence_mbar_init();
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar)) : "memory");
    mbar_wait(smem_u32(&bar), 0, D.status);   // the second arrival never comes
  }
}

// The residency calls copy small host arrays to the device in stream order, each
// through a pageable buffer on this stack rather than from the caller's array: the
// runtime stages a pageable source before cudaMemcpyAsync returns, so the caller may
// reuse its arrays at once even when they are page-locked (whose copies would
// otherwise read them later, in stream order). No heap memory is allocated.
template <typename T>
cudaError_t copy_staged(T* d_dst, const T* h_src, int n, cudaStream_t st) {
  constexpr int CHUNK = 4096 / sizeof(T);
  T buf[CHUNK];
  for (int i = 0; i < n; i += CHUNK) {
    const int m = n - i < CHUNK ? n - i : CHUNK;
    std::memcpy(buf, h_src + i, sizeof(T) * m);
    const cudaError_t e = cudaMemcpyAsync(d_dst + i, buf, sizeof(T) * m, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int launch_blocks(long long work, int threads) {
  long long b = (work + threads - 1) / threads;
  long long cap = 4ll * num_sms();
  if (b > cap) b = cap;
  return b < 1 ? 1 : (int)b;
}

}  // namespace

extern "C" {

const char* hs_status_string(hs_status s) {
  switch (s) {
    case HS_OK: return "ok";
    case HS_ERR_INVALID: return "invalid argument";
    case HS_ERR_OOM: return "out of device memory";
    case HS_ERR_CAPACITY: return "hot buffer capacity exceeded";
    case HS_ERR_CUDA: return "CUDA runtime error";
    case HS_ERR_TIMEOUT: return "device wait timed out";
    case HS_ERR_HOST_MISSING: return "selected page has no host copy";
    case HS_ERR_BAD_ID: return "page, row or token id out of range";
    case HS_ERR_BAD_WEIGHT: return "negative index-head weight";
    case HS_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation indexer";
    case HS_ERR_NOT_RESOLVED: return "replayed token is neither resident nor in the hot buffer";
    case HS_ERR_RANGE: return "attention input beyond the fp16 range of the batched path";
  }
  return "unknown status";
}

// HS_IDX_FP8 key caches as 2-D byte tensors of 128-byte rows (a page is 66 rows: 64
// keys, then 2 rows of scales); the tensor load of one page's 64 key rows lands
// 128-byte swizzled, the K-major operand layout of tcgen05.mma.
static hs_status make_key_tensor_maps(hs_pool* p, void* const* d_idx_layers) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return HS_ERR_CUDA;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  p->idx_tmaps.resize(3 * (size_t)p->d.n_groups);
  const cuuint64_t np = (cuuint64_t)p->cfg.num_idx_pages;
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int g = 0; g < p->d.n_groups; ++g) {
    CUtensorMap* m = &p->idx_tmaps[3 * (size_t)g];
    uint8_t* base = static_cast<uint8_t*>(d_idx_layers[g]);
    // one page: rows of 128 bytes over the whole cache, box of the page's 64 key rows
    const cuuint64_t dims1[2] = {128, np * (HS_IDX_FP8_PAGE_BYTES / 128)};
    const cuuint64_t str1[1] = {128};
    const cuuint32_t box1[2] = {128, (cuuint32_t)PAGE};
    // two adjacent pages: (128 bytes, 64 key rows, page), page stride 8,448 bytes
    const cuuint64_t dims2[3] = {128, (cuuint64_t)PAGE, np};
    const cuuint64_t str2[2] = {128, HS_IDX_FP8_PAGE_BYTES};
    const cuuint32_t box2[3] = {128, (cuuint32_t)PAGE, 2};
    // the 256 scale bytes of two adjacent pages
    const cuuint64_t dims3[2] = {(cuuint64_t)PAGE * 4, np};
    const cuuint64_t str3[1] = {HS_IDX_FP8_PAGE_BYTES};
    const cuuint32_t box3[2] = {(cuuint32_t)PAGE * 4, 2};
    if (encode(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims1, str1, box1, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims2, str2, box2, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&m[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base + PAGE * IDX_DIM, dims3, str3, box3, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return HS_ERR_INVALID;
  }
  return HS_OK;
}

hs_status hs_pool_config_check(const hs_pool_config* cfg) {
  if (!cfg) return HS_ERR_INVALID;
  const hs_pool_config& c = *cfg;
  if (c.page_size != PAGE || c.row_bytes != ROW || c.idx_dim != IDX_DIM) return HS_ERR_INVALID;
  if (c.n_idx_heads < 16 || c.n_idx_heads > 64 || c.n_idx_heads % 16) return HS_ERR_INVALID;
  if (c.n_heads != 16 && c.n_heads != 32 && c.n_heads != 64) return HS_ERR_INVALID;
  if (c.topk < 128 || c.topk > 2048 || c.topk % ATTN_ROWS) return HS_ERR_INVALID;
  if (c.n_layers < 1 || c.n_layers > 64 || c.layers_per_indexer < 1 || c.layers_per_indexer > 8) return HS_ERR_INVALID;
  if (c.num_pages < 1 || c.num_idx_pages < 1 || c.max_requests < 1 || c.max_ctx < 128 || c.max_ctx % 128)
    return HS_ERR_INVALID;
  if ((long long)c.num_pages * PAGE >= (1ll << 31)) return HS_ERR_INVALID;
  if (c.max_ctx > HS_MAX_CTX) return HS_ERR_INVALID;   // also keeps token ids within the 21-bit tie-break field
  if (c.max_q_per_req < 1 || c.max_q_per_req > 4 || c.max_q_per_req * c.topk > 8192) return HS_ERR_INVALID;
  if (c.max_q_per_req * c.n_idx_heads > 256) return HS_ERR_INVALID;
  if (c.hot_rows < PAGE || c.hot_rows % PAGE || c.hot_rows > 16384) return HS_ERR_INVALID;
  if (c.max_tokens < 1 || c.max_tokens > 1024 || c.host_pages < 1) return HS_ERR_INVALID;
  if (c.idx_format != HS_IDX_INT8 && c.idx_format != HS_IDX_FP8) return HS_ERR_INVALID;
  return HS_OK;
}

hs_status hs_pool_init(const hs_pool_config* cfg, void* const* d_kv_layers, void* const* d_idx_layers,
                       void* h_host_kv, hs_pool** out) {
  CallRange nvtx_range("hs_pool_init");
  if (!cfg || !d_kv_layers || !d_idx_layers || !h_host_kv || !out) return HS_ERR_INVALID;
  *out = nullptr;
  if (hs_pool_config_check(cfg) != HS_OK) return HS_ERR_INVALID;
  const hs_pool_config& c = *cfg;
  const int n_groups = (c.n_layers + c.layers_per_indexer - 1) / c.layers_per_indexer;
  for (int l = 0; l < c.n_layers; ++l)
    if (!d_kv_layers[l] || !aligned16(d_kv_layers[l])) return HS_ERR_INVALID;
  for (int g = 0; g < n_groups; ++g)
    if (!d_idx_layers[g] || !aligned16(d_idx_layers[g])) return HS_ERR_INVALID;
  void* host_dev = nullptr;
  if (cudaHostGetDevicePointer(&host_dev, h_host_kv, 0) != cudaSuccess || !aligned16(host_dev)) {
    cudaGetLastError();
    return HS_ERR_INVALID;
  }

  hs_pool* p = new (std::nothrow) hs_pool();
  if (!p) return HS_ERR_OOM;
  p->cfg = c;
  cudaGetDevice(&p->device);
  Dev& D = p->d;
  D.n_idx_heads = c.n_idx_heads;
  D.n_heads = c.n_heads;
  D.topk = c.topk;
  D.n_layers = c.n_layers;
  D.lpi = c.layers_per_indexer;
  D.n_groups = n_groups;
  D.num_pages = c.num_pages;
  D.num_idx_pages = c.num_idx_pages;
  D.max_requests = c.max_requests;
  D.max_ctx = c.max_ctx;
  D.max_pages = c.max_ctx / PAGE;
  D.max_q = c.max_q_per_req;
  D.hot_rows = c.hot_rows;
  D.hot_pages_max = c.hot_rows / PAGE;
  D.max_tokens = c.max_tokens;
  D.host_pages = c.host_pages;
  D.host = static_cast<uint8_t*>(host_dev);
  D.idx_fmt = c.idx_format;
  D.idx_page_bytes = c.idx_format == HS_IDX_FP8 ? HS_IDX_FP8_PAGE_BYTES : IDX_PAGE_BYTES;

  const size_t R = c.max_requests, P = D.max_pages, G = n_groups;
  hs_status s = HS_OK;
  auto chk = [&](hs_status x) { if (s == HS_OK) s = x; };
  chk(dev_alloc(p, &D.bt, R * P, 0xFF));
  chk(dev_alloc(p, &D.idx_bt, R * P, 0xFF));
  chk(dev_alloc(p, &D.host_pg, R * P, 0xFF));
  chk(dev_alloc(p, &D.hot_pages, R * G * D.hot_pages_max, 0xFF));
  chk(dev_alloc(p, &D.n_hot, R * G, 0));
  chk(dev_alloc(p, &D.slot_token, R * G * c.hot_rows, 0xFF));
  chk(dev_alloc(p, &D.slot_stamp, R * G * c.hot_rows, 0xFF));
  chk(dev_alloc(p, &D.tok2slot, R * G * c.max_ctx, 0xFF));
  chk(dev_alloc(p, &D.kv, (size_t)c.n_layers, 0));
  chk(dev_alloc(p, &D.idx, G, 0));
  chk(dev_alloc(p, &D.status, 1, 0));
  chk(dev_alloc(p, &D.counters, (size_t)C_N, 0));
  chk(dev_alloc(p, &D.scores, (size_t)c.max_tokens * c.max_ctx, 0));
  chk(dev_alloc(p, &D.o_part, (size_t)c.max_tokens * MAX_SPLITS * 512 * 64, 0));
  chk(dev_alloc(p, &D.o_stats, (size_t)c.max_tokens * MAX_SPLITS * 64, 0));
  {
    const int g_min = sel_wide_min_g(c.max_ctx);
    int tok = num_sms() / g_min;
    if (tok > c.max_tokens) tok = c.max_tokens;
    D.sel_ws_tokens = tok;
    chk(dev_alloc(p, &D.sel_ws, (size_t)(tok > 0 ? tok : 1) * sizeof(SelWs), 0));
    D.bsel_tokens = c.max_tokens < BS_MAX_TOKENS ? c.max_tokens : BS_MAX_TOKENS;
    chk(dev_alloc(p, &D.bsel, (size_t)D.bsel_tokens * sizeof(BselTok), 0));
  }
  if (s == HS_OK) {
    if (cudaMemcpy(D.kv, d_kv_layers, sizeof(void*) * c.n_layers, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(D.idx, d_idx_layers, sizeof(void*) * n_groups, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      s = HS_ERR_CUDA;
  }
  if (s == HS_OK && c.idx_format == HS_IDX_FP8) s = make_key_tensor_maps(p, d_idx_layers);
  if (s != HS_OK) {
    hs_pool_destroy(p);
    return s;
  }
  p->n_hot_host.assign(R * G, 0);
  *out = p;
  return HS_OK;
}

hs_status hs_pool_destroy(hs_pool* pool) {
  CallRange nvtx_range("hs_pool_destroy");
  if (!pool) return HS_ERR_INVALID;
  cudaDeviceSynchronize();
  for (void* a : pool->allocations) cudaFree(a);
  delete pool;
  return HS_OK;
}

hs_status hs_request_set_pages(hs_pool* p, int32_t req, int32_t first_page, int32_t n, const int32_t* h_block_table,
                               const int32_t* h_idx_pages, const int64_t* h_host_pages, hs_stream_t stream) {
  CallRange nvtx_range("hs_request_set_pages");
  if (!p || req < 0 || req >= p->cfg.max_requests || first_page < 0 || n < 0 ||
      (long long)first_page + n > p->d.max_pages)
    return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t off = (size_t)req * p->d.max_pages + first_page;
  for (int i = 0; i < n; ++i) {
    if (h_block_table && (h_block_table[i] < -1 || h_block_table[i] >= p->cfg.num_pages)) return HS_ERR_INVALID;
    if (h_idx_pages && (h_idx_pages[i] < -1 || h_idx_pages[i] >= p->cfg.num_idx_pages)) return HS_ERR_INVALID;
    if (h_host_pages && (h_host_pages[i] < -1 || h_host_pages[i] >= p->cfg.host_pages)) return HS_ERR_INVALID;
  }
  if (h_block_table) HS_CUDA_TRY(copy_staged(p->d.bt + off, h_block_table, n, st));
  if (h_idx_pages) HS_CUDA_TRY(copy_staged(p->d.idx_bt + off, h_idx_pages, n, st));
  if (h_host_pages) HS_CUDA_TRY(copy_staged(p->d.host_pg + off, h_host_pages, n, st));
  return HS_OK;
}

hs_status hs_hot_lease(hs_pool* p, int32_t req, int32_t group, int32_t n, const int32_t* h_pool_pages,
                       hs_stream_t stream) {
  CallRange nvtx_range("hs_hot_lease");
  if (!p || req < 0 || req >= p->cfg.max_requests || group < 0 || group >= p->d.n_groups || n < 0 ||
      (n > 0 && !h_pool_pages))
    return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  const size_t rg = (size_t)req * p->d.n_groups + group;
  const int cur = p->n_hot_host[rg];
  if (cur + n > p->d.hot_pages_max) return HS_ERR_INVALID;
  for (int i = 0; i < n; ++i)
    if (h_pool_pages[i] < 0 || h_pool_pages[i] >= p->cfg.num_pages) return HS_ERR_INVALID;
  if (n == 0) return HS_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  HS_CUDA_TRY(copy_staged(p->d.hot_pages + rg * p->d.hot_pages_max + cur, h_pool_pages, n, st));
  p->n_hot_host[rg] = cur + n;
  HS_CUDA_TRY(cudaMemcpyAsync(p->d.n_hot + rg, &p->n_hot_host[rg], sizeof(int32_t), cudaMemcpyHostToDevice, st));
  return HS_OK;
}

hs_status hs_hot_release(hs_pool* p, int32_t req, hs_stream_t stream) {
  CallRange nvtx_range("hs_hot_release");
  if (!p || req < 0 || req >= p->cfg.max_requests) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  clear_hot_kernel<<<launch_blocks(p->cfg.max_ctx, 256), 256, 0, st>>>(p->d, req);
  HS_CUDA_TRY(cudaGetLastError());
  for (int g = 0; g < p->d.n_groups; ++g) p->n_hot_host[(size_t)req * p->d.n_groups + g] = 0;
  return HS_OK;
}

hs_status hs_append_rows(hs_pool* p, int32_t n, const int32_t* d_req, const int32_t* d_pos, const uint8_t* d_kv_rows,
                         const int8_t* d_idx_keys, hs_stream_t stream) {
  CallRange nvtx_range("hs_append_rows");
  if (!p || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  if (!d_req || !d_pos || !d_kv_rows || !d_idx_keys || !aligned16(d_kv_rows) || !aligned16(d_idx_keys))
    return HS_ERR_INVALID;
  const long long work = (long long)n * (p->d.n_layers * ROW_CHUNKS + p->d.n_groups * (IDX_DIM / 16));
  return launch_pdl(append_kernel, dim3(launch_blocks(work, 256)), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                    0, p->d, n, d_req, d_pos, d_kv_rows, d_idx_keys);
}

hs_status hs_indexer_topk(hs_pool* p, int32_t index_layer, int32_t n, const int32_t* d_req, const int32_t* d_limit,
                          const int8_t* d_q, const int8_t* d_w, int32_t* d_topk, int64_t* d_scores,
                          hs_stream_t stream) {
  CallRange nvtx_range("hs_indexer_topk");
  if (!p || index_layer < 0 || index_layer >= p->d.n_groups || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  if (!d_req || !d_limit || !d_q || !d_w || !d_topk || !aligned16(d_q)) return HS_ERR_INVALID;
  if (d_scores && !aligned16(d_scores)) return HS_ERR_INVALID;
  if (p->d.idx_fmt != HS_IDX_INT8) return HS_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int64_t* scores = d_scores ? d_scores : p->d.scores;
  uint32_t* hist0 = select_hist0(p, n, true);
  hs_status s = launch_indexer(p, index_layer, n, d_req, d_limit, d_q, d_w, scores, hist0, st);
  if (s != HS_OK) return s;
  return launch_select(p, n, scores, p->cfg.max_ctx, d_limit, d_topk, st, false, true, hist0 != nullptr);
}

hs_status hs_indexer_topk_fp8(hs_pool* p, int32_t index_layer, int32_t n, const int32_t* d_req,
                              const int32_t* d_limit, const uint8_t* d_q, const float* d_w, int32_t* d_topk,
                              float* d_scores, hs_stream_t stream) {
  CallRange nvtx_range("hs_indexer_topk_fp8");
  if (!p || index_layer < 0 || index_layer >= p->d.n_groups || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  if (p->d.idx_fmt != HS_IDX_FP8) return HS_ERR_INVALID;
  if (!d_req || !d_limit || !d_q || !d_w || !d_topk || !aligned16(d_q) || (reinterpret_cast<uintptr_t>(d_w) & 3))
    return HS_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the kernel writes each score as an order-preserving integer for the selection
  uint32_t* hist0 = select_hist0(p, n, true);
  hs_status s = launch_indexer_fp8(p, index_layer, n, d_req, d_limit, d_q, d_w, p->d.scores, d_scores, hist0, st);
  if (s != HS_OK) return s;
  return launch_select(p, n, p->d.scores, p->cfg.max_ctx, d_limit, d_topk, st, true, true, hist0 != nullptr);
}

hs_status hs_resolve_topk(hs_pool* p, int32_t group, int32_t step, int32_t n, const int32_t* d_req,
                          const int32_t* d_topk, int32_t* d_row_ids, hs_plan_entry* d_plan, hs_stream_t stream) {
  CallRange nvtx_range("hs_resolve_topk");
  if (!p || group < 0 || group >= p->d.n_groups || step < 0 || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  if (!d_req || !d_topk || !d_row_ids) return HS_ERR_INVALID;
  return launch_resolve(p, group, step, n, d_req, d_topk, d_row_ids, d_plan, reinterpret_cast<cudaStream_t>(stream));
}

hs_status hs_replay_topk(hs_pool* p, int32_t group, int32_t n, const int32_t* d_req, const int32_t* d_topk,
                         int32_t* d_row_ids, hs_stream_t stream) {
  CallRange nvtx_range("hs_replay_topk");
  if (!p || group < 0 || group >= p->d.n_groups || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  if (!d_req || !d_topk || !d_row_ids) return HS_ERR_INVALID;
  return launch_replay(p, group, n, d_req, d_topk, d_row_ids, reinterpret_cast<cudaStream_t>(stream));
}

hs_status hs_sparse_mla_decode(hs_pool* p, int32_t layer, int32_t n, const uint16_t* d_q, const int32_t* d_row_ids,
                               float sm_scale, uint16_t* d_out, float* d_lse, hs_stream_t stream) {
  CallRange nvtx_range("hs_sparse_mla_decode");
  if (!p || layer < 0 || layer >= p->cfg.n_layers || n < 0 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  if (n == 0) return HS_OK;
  if (!d_q || !d_row_ids || !d_out || !aligned16(d_q) || !aligned16(d_out)) return HS_ERR_INVALID;
  // the previous launch of this pool was a decode over the same rows on this stream:
  // the row ids and rows are final before that kernel started
  const bool settled = p->settled_rows == d_row_ids && p->settled_stream == stream;
  const hs_status s = launch_attention(p, layer, n, d_q, d_row_ids, sm_scale, d_out, d_lse, settled,
                                       reinterpret_cast<cudaStream_t>(stream));
  p->settled_rows = s == HS_OK ? d_row_ids : nullptr;
  p->settled_stream = stream;
  return s;
}

hs_status hs_offload_pages(hs_pool* p, int32_t n, const int32_t* d_pool_pages, const int64_t* d_host_pages,
                           hs_stream_t stream) {
  CallRange nvtx_range("hs_offload_pages");
  if (!p || n < 0) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  if (n == 0) return HS_OK;
  if (!d_pool_pages || !d_host_pages) return HS_ERR_INVALID;
  const long long work = (long long)n * p->d.n_layers * (PAGE * ROW / 16);
  return launch_pdl(offload_kernel, dim3(launch_blocks(work, 256)), dim3(256), 0,
                    reinterpret_cast<cudaStream_t>(stream), 0, p->d, n, d_pool_pages, d_host_pages);
}

hs_status hs_link_probe(const void* h_mapped, int64_t n_host_rows, int32_t row_bytes, const int64_t* d_src_rows,
                        int64_t n, void* d_dst, hs_stream_t stream) {
  CallRange nvtx_range("hs_link_probe");
  if (!h_mapped || !d_src_rows || !d_dst || n < 0 || n_host_rows < 1 || row_bytes < 16 || row_bytes % 16 ||
      !aligned16(d_dst) || !aligned16(h_mapped))
    return HS_ERR_INVALID;
  if (n == 0) return HS_OK;
  void* src = nullptr;
  if (cudaHostGetDevicePointer(&src, const_cast<void*>(h_mapped), 0) != cudaSuccess || !aligned16(src)) {
    cudaGetLastError();
    return HS_ERR_INVALID;
  }
  const long long work = n * (row_bytes / 16);
  link_probe_kernel<<<launch_blocks((work + 3) / 4, 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(src), n_host_rows, row_bytes, d_src_rows, n, static_cast<uint8_t*>(d_dst));
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

hs_status hs_wait_selftest(hs_pool* p, hs_stream_t stream) {
  CallRange nvtx_range("hs_wait_selftest");
  if (!p) return HS_ERR_INVALID;
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p->d);
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

hs_status hs_select_selftest(hs_pool* p, int32_t n, const int32_t* d_limit, int32_t* d_topk, hs_stream_t stream) {
  CallRange nvtx_range("hs_select_selftest");
  if (!p || !d_limit || !d_topk || n < 1 || n > p->cfg.max_tokens) return HS_ERR_INVALID;
  const int G = select_wide_groups(p, n, true);
  if (G == 0) return HS_ERR_INVALID;
  p->settled_rows = nullptr;
  return launch_select_wide(p, n, p->d.scores, p->cfg.max_ctx, d_limit, d_topk, p->d.idx_fmt == HS_IDX_FP8, G, false,
                            reinterpret_cast<cudaStream_t>(stream), true);
}

hs_status hs_get_error(hs_pool* p, hs_status* device_status, hs_stream_t stream) {
  CallRange nvtx_range("hs_get_error");
  if (!p || !device_status) return HS_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  HS_CUDA_TRY(cudaStreamSynchronize(st));
  int32_t v = 0;
  HS_CUDA_TRY(cudaMemcpy(&v, p->d.status, sizeof(v), cudaMemcpyDeviceToHost));
  HS_CUDA_TRY(cudaMemset(p->d.status, 0, sizeof(int32_t)));
  if (v == HS_ERR_TIMEOUT && p->d.sel_ws) {
    // a grid-wide wait of the selection may have given up half way: start its scratch
    // (arrival counters, histogram sums, candidate list, the flag that routes later
    // selections around it) from zero again
    HS_CUDA_TRY(cudaMemset(p->d.sel_ws, 0, (size_t)p->d.sel_ws_tokens * sizeof(SelWs)));
    HS_CUDA_TRY(cudaDeviceSynchronize());
  }
  *device_status = static_cast<hs_status>(v);
  return HS_OK;
}

hs_status hs_set_select_mode(hs_pool* p, int32_t mode) {
  CallRange nvtx_range("hs_set_select_mode");
  if (!p || (mode != HS_SELECT_AUTO && mode != HS_SELECT_LOCAL)) return HS_ERR_INVALID;
  p->select_mode = mode;
  return HS_OK;
}

hs_status hs_get_counters(hs_pool* p, hs_counters* out, int32_t reset, hs_stream_t stream) {
  CallRange nvtx_range("hs_get_counters");
  if (!p || !out) return HS_ERR_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  HS_CUDA_TRY(cudaStreamSynchronize(st));
  unsigned long long v[C_N];
  HS_CUDA_TRY(cudaMemcpy(v, p->d.counters, sizeof(v), cudaMemcpyDeviceToHost));
  std::memset(out, 0, sizeof(*out));
  out->resident = v[C_RESIDENT];
  out->hits = v[C_HITS];
  out->misses = v[C_MISSES];
  out->h2d_bytes = v[C_H2D];
  out->d2h_bytes = v[C_D2H];
  if (reset) HS_CUDA_TRY(cudaMemset(p->d.counters, 0, sizeof(v)));
  return HS_OK;
}

}  // extern "C"
