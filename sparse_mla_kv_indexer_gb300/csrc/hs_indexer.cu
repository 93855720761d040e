// Indexer scoring and top-K selection for one indexer layer.
//
// "Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse" (vLLM blog Part 2),
// section "Why not TP or DP?": the indexer scores every earlier token so sparse
// MLA can pick the 2,048 it attends to. Integer form used here:
//   s[t] = sum_h w[h] * max(0, sum_d q[h][d] * k_t[d]),  int8 in, exact int64 out.
//
// Scoring kernel (one persistent CTA per SM):
//  * work item = (request segment, 128-key tile); the T <= 4 query tokens of a
//    request share each key tile, so the keys are read from HBM once per request;
//  * key pages (64 x 128 B) arrive by bulk copy (TMA unit) into a 4-stage ring
//    filled by a producer warp; converter warps, an MMA warp and epilogue warps
//    work on consecutive tiles at once (double-buffered A tiles and accumulators);
//  * int8 keys and queries are widened to fp16 (exact for |x| <= 128) in the
//    128-byte-swizzled K-major layout and contracted on the tensor cores with
//    tcgen05.mma kind::f16 (M = 128 keys, N = T * H_i, K = 128); the products
//    and 128-term sums are integers below 2^24, exact in the fp32 accumulator;
//  * the epilogue reads the accumulator from tensor memory, applies ReLU and
//    the head weights in integer arithmetic and writes int64 scores.
//
// Select kernel (one 8- or 16-CTA cluster per query token): a shared-memory
// histogram of a monotone bucket of each (score, token) key, merged through
// distributed shared memory, finds the bucket of the K-th largest; the few keys
// in that bucket are sorted by the cluster leader to give the exact threshold
// key (a multi-level histogram refinement takes over when a bucket is crowded);
// each CTA then emits its selected tokens in ascending order at its offset.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {

// ----------------------------------------------------------------------------------
// Scoring kernel
// ----------------------------------------------------------------------------------
// Warp roles (320 threads):
//   warps 0-3  epilogue: TMEM accumulator -> ReLU, head weights, int64 scores
//   warps 4-7  convert: raw int8 key tile -> fp16 A tile; queries -> fp16 B operand
//   warp 8     producer: bulk copies of key pages into a 4-stage ring
//   warp 9     MMA issuer: tcgen05.mma into one of two TMEM accumulators
constexpr int IX_THREADS = 320;
constexpr int IX_STAGES = 4;
constexpr int IX_TILE = 128;
constexpr int IX_RAW = IX_TILE * IDX_DIM;              // 16 KB int8 per tile
constexpr int IX_A_COL = IX_TILE * 128;                // one 64-dim fp16 atom column, 16 KB
constexpr int IX_A = 2 * IX_A_COL;                     // 32 KB per A tile
constexpr int IX_B_COL = 256 * 128;                    // B atom column for up to N = 256 rows
constexpr int IX_MAX_SEG = 1024;
constexpr int IX_OFF_A = 0;                            // 2 A tiles
constexpr int IX_OFF_B = IX_OFF_A + 2 * IX_A;          // 64 KB
constexpr int IX_OFF_RAW = IX_OFF_B + 2 * IX_B_COL;    // 128 KB
constexpr int IX_OFF_BAR = IX_OFF_RAW + IX_STAGES * IX_RAW;   // 192 KB
constexpr int IX_OFF_SEG = IX_OFF_BAR + 256;
constexpr int IX_SMEM = IX_OFF_SEG + IX_MAX_SEG * 16 + 4 * 64 * 4 + 2 * IX_MAX_SEG * 4 + 1024;
constexpr int IX_TMEM_COLS = 512;                      // two accumulators of up to 256 columns

struct IxSeg {
  int32_t first;     // first token of the segment
  int32_t ntok;      // tokens in the segment
  int32_t maxlim;    // max causal limit over its tokens
  int32_t tile_end;  // exclusive prefix of tiles
};

// widen 4 packed int8 to 4 fp16 (exact): 0x64XX as fp16 is 1024 + XX
__device__ __forceinline__ uint2 i8x4_to_f16x4(uint32_t x) {
  uint32_t u = x ^ 0x80808080u;
  uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 a = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
  __half2 b = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
  return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

// 16 int8 (one uint4) -> two 16-byte fp16 chunks
__device__ __forceinline__ void i8x16_to_f16(uint4 v, uint4& c0, uint4& c1) {
  uint2 a = i8x4_to_f16x4(v.x), b = i8x4_to_f16x4(v.y), c = i8x4_to_f16x4(v.z), d = i8x4_to_f16x4(v.w);
  c0 = make_uint4(a.x, a.y, b.x, b.y);
  c1 = make_uint4(c.x, c.y, d.x, d.y);
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(IX_THREADS, 1)
indexer_kernel(Dev D, int il, int n_tok, const int32_t* __restrict__ req_of, const int32_t* __restrict__ limit_of,
               const int8_t* __restrict__ qg, const int8_t* __restrict__ wg, int64_t* __restrict__ scores,
               int ld) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + IX_OFF_BAR);
  uint64_t* raw_full = bars;                      // [4]
  uint64_t* raw_empty = bars + 4;                 // [4]
  uint64_t* a_full = bars + 8;                    // [2]
  uint64_t* a_empty = bars + 10;                  // [2]
  uint64_t* t_full = bars + 12;                   // [2]
  uint64_t* t_empty = bars + 14;                  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  int32_t* s_nseg = reinterpret_cast<int32_t*>(tmem_slot + 1);
  int32_t* s_dead = s_nseg + 1;
  int32_t* s_issued = s_nseg + 2;
  int32_t* s_consumed = s_nseg + 3;
  IxSeg* segs = reinterpret_cast<IxSeg*>(smem + IX_OFF_SEG);
  int32_t* s_w = reinterpret_cast<int32_t*>(smem + IX_OFF_SEG + IX_MAX_SEG * 16);   // [4][64], epilogue-owned
  int32_t* s_req = s_w + 4 * 64;                                                      // [n_tok]
  int32_t* s_lim = s_req + IX_MAX_SEG;                                                // [n_tok]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hi = D.n_idx_heads;
  const int8_t* keys = D.idx[il];

  // ---- request segments of the batch (tokens of one request are contiguous) ----
  for (int t = tid; t < n_tok; t += IX_THREADS) {
    int r = req_of[t], lim = limit_of[t];
    if (r < 0 || r >= D.max_requests || lim < 0 || lim > D.max_ctx || lim > ld) {
      set_status(D.status, HS_ERR_BAD_ID);
      r = 0;
      lim = 0;
    }
    s_req[t] = r;
    s_lim[t] = lim;
  }
  __syncthreads();
  if (tid == 0) {
    int ns = 0, tiles = 0;
    for (int t = 0; t < n_tok; ++t) {
      if (t == 0 || s_req[t] != s_req[t - 1] || segs[ns - 1].ntok == D.max_q) {
        segs[ns].first = t;
        segs[ns].ntok = 0;
        segs[ns].maxlim = 0;
        ++ns;
      }
      IxSeg& sgm = segs[ns - 1];
      sgm.ntok++;
      sgm.maxlim = max(sgm.maxlim, s_lim[t]);
    }
    for (int i = 0; i < ns; ++i) {
      tiles += (segs[i].maxlim + IX_TILE - 1) / IX_TILE;
      segs[i].tile_end = tiles;
    }
    *s_nseg = ns;
    for (int b = 0; b < 16; ++b) mbar_init(smem_u32(&bars[b]), 1);
    fence_mbar_init();
    *s_dead = 0;
    *s_issued = 0;
    *s_consumed = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), IX_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nseg = *s_nseg;
  const int total = nseg ? segs[nseg - 1].tile_end : 0;
  const int n_local = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  auto seg_of = [&](int item) {
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (segs[mid].tile_end > item) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  auto item_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };

  if (warp == 8) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      for (int i = 0; i < n_local; ++i) {
        const int rs = i % IX_STAGES;
        if (i >= IX_STAGES && !mbar_wait(smem_u32(&raw_empty[rs]), ((i / IX_STAGES) - 1) & 1, D.status)) {
          *s_dead = 1;
          break;
        }
        if (*(volatile int32_t*)s_dead) break;
        const int item = item_of(i);
        const int sg = seg_of(item);
        const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
        const int r = s_req[segs[sg].first];
        const uint32_t bar = smem_u32(&raw_full[rs]);
        const uint32_t dst = smem_u32(smem + IX_OFF_RAW + rs * IX_RAW);
        const int npg = ((tile * IX_TILE + PAGE) < segs[sg].maxlim) ? 2 : 1;
        int ip[2] = {-1, -1};
        uint32_t bytes = 0;
        for (int k = 0; k < npg; ++k) {
          int v = D.idx_bt[(size_t)r * D.max_pages + tile * 2 + k];
          if (v < 0 || v >= D.num_idx_pages) { set_status(D.status, HS_ERR_BAD_ID); continue; }
          ip[k] = v;
          bytes += IDX_PAGE_BYTES;
        }
        mbar_expect_tx(bar, bytes);
        for (int k = 0; k < 2; ++k)
          if (ip[k] >= 0) bulk_g2s(dst + k * IDX_PAGE_BYTES, keys + (size_t)ip[k] * IDX_PAGE_BYTES, IDX_PAGE_BYTES, bar);
        *s_issued = i + 1;
      }
    }
  } else if (warp == 9) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      for (int i = 0; i < n_local; ++i) {
        const int ab = i & 1;
        if (!mbar_wait(smem_u32(&a_full[ab]), (i >> 1) & 1, D.status)) { *s_dead = 1; break; }
        if (i >= 2 && !mbar_wait(smem_u32(&t_empty[ab]), ((i >> 1) - 1) & 1, D.status)) { *s_dead = 1; break; }
        if (*(volatile int32_t*)s_dead) break;
        tc_fence_after();
        const IxSeg S = segs[seg_of(item_of(i))];
        const int N = ((S.ntok * Hi) + 15) & ~15;
        const uint32_t idesc = idesc_f16(128, N, false, false);
        const uint32_t a0 = smem_u32(smem + IX_OFF_A + ab * IX_A), b0 = smem_u32(smem + IX_OFF_B);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * IX_A_COL + (kk & 3) * 32, 16, 1024);
          uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * IX_B_COL + (kk & 3) * 32, 16, 1024);
          umma_f16(tmem + ab * 256, ad, bd, idesc, kk > 0);
        }
        umma_commit(smem_u32(&a_empty[ab]));
        umma_commit(smem_u32(&t_full[ab]));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------ converters ------------------------------
    const int ct = tid - 128;
    int cur_seg = -1;
    for (int i = 0; i < n_local; ++i) {
      const int item = item_of(i);
      const int sg = seg_of(item);
      const IxSeg S = segs[sg];
      const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
      const int key0 = tile * IX_TILE;
      bool ok = true;
      if (sg != cur_seg) {
        // every MMA reading the previous queries has completed before they are replaced
        if (i > 0) ok = mbar_wait(smem_u32(&a_empty[(i - 1) & 1]), ((i - 1) >> 1) & 1, D.status);
        uint8_t* B = smem + IX_OFF_B;
        const int N = ((S.ntok * Hi) + 15) & ~15;
        for (int c = ct; c < N * 8; c += 128) {
          const int row = c >> 3, ch16 = c & 7;       // 8 chunks of 16 int8 per 128-dim row
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < S.ntok * Hi) {
            const int j = row / Hi, h = row - j * Hi;
            v = *reinterpret_cast<const uint4*>(qg + ((size_t)(S.first + j) * Hi + h) * IDX_DIM + ch16 * 16);
          }
          uint4 c0, c1;
          i8x16_to_f16(v, c0, c1);
          const int dim0 = ch16 * 16;
          uint8_t* base = B + (dim0 >> 6) * IX_B_COL;
          const int chunk = (dim0 & 63) >> 3;
          *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk)) = c0;
          *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk + 1)) = c1;
        }
        cur_seg = sg;
      }
      const int rs = i % IX_STAGES, ab = i & 1;
      if (ok) ok = mbar_wait(smem_u32(&raw_full[rs]), (i / IX_STAGES) & 1, D.status);
      if (ok && i >= 2) ok = mbar_wait(smem_u32(&a_empty[ab]), ((i >> 1) - 1) & 1, D.status);
      if (!ok) *s_dead = 1;
      const uint8_t* raw = smem + IX_OFF_RAW + rs * IX_RAW;
      uint8_t* A = smem + IX_OFF_A + ab * IX_A;
      for (int c = ct; c < IX_TILE * 8; c += 128) {
        const int row = c >> 3, ch16 = c & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (key0 + row < S.maxlim) v = *reinterpret_cast<const uint4*>(raw + row * IDX_DIM + ch16 * 16);
        uint4 c0, c1;
        i8x16_to_f16(v, c0, c1);
        const int dim0 = ch16 * 16;
        uint8_t* base = A + (dim0 >> 6) * IX_A_COL;
        const int chunk = (dim0 & 63) >> 3;
        *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk)) = c0;
        *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk + 1)) = c1;
      }
      fence_proxy_async();
      named_sync(1, 128);
      if (ct == 0) {
        *s_consumed = i + 1;
        mbar_arrive(smem_u32(&raw_empty[rs]));
        mbar_arrive(smem_u32(&a_full[ab]));
      }
      if (*(volatile int32_t*)s_dead) break;
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    int cur_seg = -1;
    for (int i = 0; i < n_local; ++i) {
      const int item = item_of(i);
      const int sg = seg_of(item);
      const IxSeg S = segs[sg];
      const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
      const int key = tile * IX_TILE + warp * 32 + lane;
      if (sg != cur_seg) {
        named_sync(2, 128);
        for (int c = tid; c < 4 * 64; c += 128) {
          const int j = c >> 6, h = c & 63;
          int w = 0;
          if (j < S.ntok && h < Hi) {
            w = wg[(size_t)(S.first + j) * Hi + h];
            if (w < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); w = 0; }
          }
          s_w[c] = w;
        }
        named_sync(2, 128);
        cur_seg = sg;
      }
      const int ab = i & 1;
      if (!mbar_wait(smem_u32(&t_full[ab]), (i >> 1) & 1, D.status)) { *s_dead = 1; break; }
      tc_fence_after();
      for (int j = 0; j < S.ntok; ++j) {
        const int lim = s_lim[S.first + j];
        long long acc = 0;
        for (int h0 = 0; h0 < Hi; h0 += 16) {
          uint32_t r[16];
          tmem_ld16(lane_base + (uint32_t)(ab * 256 + j * Hi + h0), r);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int v = max(__float2int_rn(__uint_as_float(r[k])), 0);
            acc += (long long)v * s_w[j * 64 + h0 + k];
          }
        }
        if (key < lim) scores[(size_t)(S.first + j) * ld + key] = acc;
      }
      tc_fence_before();
      named_sync(2, 128);
      if (tid == 0) mbar_arrive(smem_u32(&t_empty[ab]));
      if (*(volatile int32_t*)s_dead) break;
    }
  }
  __syncthreads();
  if (*s_dead && tid == 8 * 32) {
    // drain bulk copies still in flight before the CTA's shared memory goes away
    for (int k = *s_consumed; k < *s_issued; ++k)
      mbar_wait(smem_u32(&raw_full[k % IX_STAGES]), (k / IX_STAGES) & 1, D.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, IX_TMEM_COLS);
}

// ----------------------------------------------------------------------------------
// Select kernel
// ----------------------------------------------------------------------------------
// Each score s of token index t is made unique and order-preserving as the key
//   key = s * 2^21 + (2^21 - 1 - t)          (s >= 0, t < 2^21)
// so the top K by (score desc, token asc) are exactly the K largest keys, and the
// K-th largest key tau selects them with the single test key >= tau.
constexpr int SEL_THREADS = 512;
constexpr int SEL_BINS = 4096;
constexpr int SEL_CACHE = 20480;                       // keys cached in shared memory per CTA
constexpr int SEL_CAND = 2048;                         // candidates per CTA on the fast path
constexpr int SEL_LEAD = 4096;                         // candidates the cluster leader sorts
constexpr int SEL_SMEM = SEL_CACHE * 8 + SEL_LEAD * 8 + 1024;
constexpr unsigned long long IDX_MASK = (1ull << 21) - 1;

// monotone level-0 bucket of a key: exact below 64, then 64 buckets per octave
__device__ __forceinline__ int bucket1(unsigned long long v) {
  if (v < 64) return (int)v;
  int e = 63 - __clzll((long long)v);
  int m = (int)((v >> (e - 6)) & 63);
  return 64 + (e - 6) * 64 + m;
}

// warp-aggregated shared-memory histogram increment
__device__ __forceinline__ void hist_add(uint32_t* hist, int bin) {
  const unsigned act = __activemask();
  const unsigned peers = __match_any_sync(act, bin);
  if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) warp_tot[lane] = t;
    if (lane == nw - 1 && total) *total = t;
  }
  __syncthreads();
  int res = x - v + (warp ? warp_tot[warp - 1] : 0);
  __syncthreads();
  return res;
}

// descending bitonic sort of n (power of two) keys
__device__ void bitonic_desc(unsigned long long* a, int n) {
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int p = i ^ j;
        if (p > i) {
          unsigned long long x = a[i], y = a[p];
          bool desc = (i & k) == 0;
          if ((x < y) == desc) { a[i] = y; a[p] = x; }
        }
      }
      __syncthreads();
    }
}

__global__ void __launch_bounds__(SEL_THREADS, 1)
select_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
              int32_t* __restrict__ topk) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int slice = SEL_BINS / CL;
  const int tok = blockIdx.x / CL;
  const int K = D.topk;
  const int tid = threadIdx.x;
  __shared__ uint32_t hist[SEL_BINS];      // level histograms; later the candidate list
  __shared__ uint32_t tot[SEL_BINS / 8];
  __shared__ int warp_tot[32];
  __shared__ int s_sum, s_bin, s_ncand, s_over, s_nsel;
  __shared__ long long s_above;
  __shared__ unsigned long long s_tau;
  extern __shared__ __align__(16) uint8_t sel_dyn[];
  unsigned long long* cache = reinterpret_cast<unsigned long long*>(sel_dyn);            // [SEL_CACHE]
  unsigned long long* lead = cache + SEL_CACHE;                                           // [SEL_LEAD]
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(hist);                 // [SEL_CAND]
  int32_t* elist = reinterpret_cast<int32_t*>(lead);                                      // [K] after tau

  int n = limit_of[tok];
  n = max(0, min(n, D.max_ctx));
  int32_t* out = topk + (size_t)tok * K;
  if (n <= K) {           // every earlier token is selected (uniform across the cluster)
    if (crank == 0)
      for (int i = tid; i < K; i += blockDim.x) out[i] = i < n ? i : -1;
    return;
  }
  const long long* s = reinterpret_cast<const long long*>(scores) + (size_t)tok * ld;
  const int per = (n + CL - 1) / CL;
  const int lo = crank * per, hi = min(n, lo + per);
  const int cnt_local = max(0, hi - lo);
  const bool cached = per <= SEL_CACHE;
  auto key_at = [&](int i) -> unsigned long long {
    if (cached) return cache[i];
    long long v = s[lo + i];
    return ((unsigned long long)max(v, 0ll) << 21) | (IDX_MASK - (unsigned long long)(lo + i));
  };

  // ---- level 0: histogram of bucket1(key); find the bucket of the K-th largest ----
  for (int b = tid; b < SEL_BINS; b += blockDim.x) hist[b] = 0;
  if (tid == 0) { s_ncand = 0; s_over = 0; s_bin = 0; s_above = 0; }
  __syncthreads();
  for (int i = tid; i < cnt_local; i += blockDim.x) {
    long long v = s[lo + i];
    if (v < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); v = 0; }
    const unsigned long long k = ((unsigned long long)v << 21) | (IDX_MASK - (unsigned long long)(lo + i));
    if (cached) cache[i] = k;
    hist_add(hist, bucket1(k));
  }
  int need = K;
  auto cluster_find = [&](void) {
    cluster.sync();
    for (int b = tid; b < slice; b += blockDim.x) {
      uint32_t a = 0;
      for (int r = 0; r < CL; ++r) a += cluster.map_shared_rank(hist, r)[crank * slice + b];
      tot[b] = a;
    }
    cluster.sync();
    for (int b = tid; b < SEL_BINS; b += blockDim.x) hist[b] = cluster.map_shared_rank(tot, b / slice)[b % slice];
    if (tid == 0) { s_bin = 0; s_above = 0; }
    __syncthreads();
    const int per_t = SEL_BINS / SEL_THREADS;     // 8 bins per thread, thread 0 = top bins
    int local = 0;
    for (int k = 0; k < per_t; ++k) local += hist[SEL_BINS - 1 - (tid * per_t + k)];
    int before = block_excl_scan(local, warp_tot, nullptr);
    if (before < need && need <= before + local) {
      int cum = before;
      for (int k = 0; k < per_t; ++k) {
        int b = SEL_BINS - 1 - (tid * per_t + k);
        if (cum + (int)hist[b] >= need) { s_bin = b; s_above = cum; break; }
        cum += hist[b];
      }
    }
    __syncthreads();
  };
  cluster_find();
  const int B0 = s_bin;
  need -= (int)s_above;
  cluster.sync();           // every CTA is done reading peers' tot[] / hist[] of level 0

  // ---- fast path: collect the keys of bucket B0, the leader sorts them ----
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  for (int i = tid; i < cnt_local; i += blockDim.x) {
    const unsigned long long k = key_at(i);
    if (bucket1(k) == B0) {
      int at = atomicAdd(&s_ncand, 1);
      if (at < SEL_CAND) cand[at] = k; else s_over = 1;
    }
  }
  cluster.sync();
  int total_c = 0, over = 0;
  for (int r = 0; r < CL; ++r) {
    total_c += min(*cluster.map_shared_rank(&s_ncand, r), SEL_CAND + 1);
    over |= *cluster.map_shared_rank(&s_over, r);
  }
  const bool fast = !over && total_c <= SEL_LEAD;
  unsigned long long tau;
  if (fast) {
    if (crank == 0) {
      int np = 1;
      while (np < total_c) np <<= 1;
      int base = 0;
      for (int r = 0; r < CL; ++r) {
        const int c = *cluster.map_shared_rank(&s_ncand, r);
        const unsigned long long* pc = cluster.map_shared_rank(cand, r);
        for (int i = tid; i < c; i += blockDim.x) lead[base + i] = pc[i];
        base += c;
      }
      for (int i = total_c + tid; i < np; i += blockDim.x) lead[i] = 0ull;
      __syncthreads();
      bitonic_desc(lead, np);
      if (tid == 0) s_tau = lead[need - 1];
    }
    cluster.sync();
    tau = *cluster.map_shared_rank(&s_tau, 0);
  } else {
    // ---- slow path (crowded bucket): refine the key range level by level ----
    unsigned long long base, width;
    if (B0 < 64) { base = B0; width = 1; }
    else {
      int e = (B0 - 64) / 64 + 6, m = (B0 - 64) % 64;
      base = (1ull << e) + ((unsigned long long)m << (e - 6));
      width = 1ull << (e - 6);
    }
    while (width > 1) {
      const int lw = 63 - __clzll((long long)width);
      const int shift = lw > 12 ? lw - 12 : 0;
      for (int b = tid; b < SEL_BINS; b += blockDim.x) hist[b] = 0;
      __syncthreads();
      for (int i = tid; i < cnt_local; i += blockDim.x) {
        const unsigned long long k = key_at(i);
        if (k >= base && k - base < width) hist_add(hist, (int)((k - base) >> shift));
      }
      cluster_find();
      base += (unsigned long long)s_bin << shift;
      need -= (int)s_above;
      width = 1ull << shift;
      cluster.sync();
    }
    tau = base;   // identical in every CTA of the cluster
  }

  // ---- emit: this CTA's selected tokens in ascending order, then place them ----
  constexpr int IPT = 8;
  int sel_run = 0;
  for (int t0 = 0; t0 < cnt_local; t0 += SEL_THREADS * IPT) {
    const int i0 = t0 + tid * IPT;
    int flags = 0, c = 0;
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      const int i = i0 + k;
      if (i < cnt_local && key_at(i) >= tau) { flags |= 1 << k; ++c; }
    }
    int pos = block_excl_scan(c, warp_tot, &s_sum) + sel_run;
    const int tile_tot = s_sum;
#pragma unroll
    for (int k = 0; k < IPT; ++k)
      if (flags >> k & 1) {
        if (pos < K) elist[pos] = lo + i0 + k;
        ++pos;
      }
    sel_run += tile_tot;
    __syncthreads();
  }
  if (tid == 0) s_nsel = sel_run;
  cluster.sync();
  int off = 0;
  for (int r = 0; r < crank; ++r) off += *cluster.map_shared_rank(&s_nsel, r);
  for (int i = tid; i < sel_run; i += blockDim.x) {
    if (off + i < K && i < K) out[off + i] = elist[i];
    else set_status(D.status, HS_ERR_BAD_ID);
  }
  cluster.sync();   // peers may still read this CTA's shared memory until here
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

hs_status launch_indexer(hs_pool* p, int il, int n, const int32_t* d_req, const int32_t* d_limit,
                         const int8_t* d_q, const int8_t* d_w, int64_t* d_scores, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, IX_SMEM) !=
        cudaSuccess)
      return HS_ERR_CUDA;
    attr = true;
  }
  indexer_kernel<<<num_sms(), IX_THREADS, IX_SMEM, st>>>(p->d, il, n, d_req, d_limit, d_q, d_w, d_scores,
                                                         p->cfg.max_ctx);
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

hs_status launch_select(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                        int32_t* d_topk, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return HS_ERR_CUDA;
    attr = true;
  }
  // 8 CTAs per token when their chunks fit the shared-memory cache, else 16
  const int cl = (p->cfg.max_ctx <= 8 * SEL_CACHE) ? 8 : 16;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n * cl, 1, 1);
  lc.blockDim = dim3(SEL_THREADS, 1, 1);
  lc.dynamicSmemBytes = SEL_SMEM;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, select_kernel, p->d, scores, ld, d_limit, d_topk) == cudaSuccess ? HS_OK
                                                                                                  : HS_ERR_CUDA;
}

}  // namespace hs
