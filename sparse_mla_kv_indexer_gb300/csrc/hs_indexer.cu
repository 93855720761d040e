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
//  * key pages (64 x 128 B) arrive by bulk copy (TMA unit) into a 6-stage ring;
//  * int8 keys and queries are widened to fp16 (exact for |x| <= 128) in the
//    128-byte-swizzled K-major layout and contracted on the tensor cores with
//    tcgen05.mma kind::f16 (M = 128 keys, N = T * H_i, K = 128); the products
//    and 128-term sums are integers below 2^24, exact in the fp32 accumulator;
//  * the epilogue reads the accumulator from tensor memory, applies ReLU and
//    the head weights in integer arithmetic and writes int64 scores.
//
// Select kernel (one 8-CTA cluster per query token): exact radix select of the
// K-th largest score using shared-memory histograms merged through distributed
// shared memory, then an ordered compaction that emits the selected token ids
// in ascending order with ties broken toward the lower token index.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {

// ----------------------------------------------------------------------------------
// Scoring kernel
// ----------------------------------------------------------------------------------
constexpr int IX_THREADS = 256;
constexpr int IX_STAGES = 6;
constexpr int IX_TILE = 128;
constexpr int IX_RAW = IX_TILE * IDX_DIM;              // 16 KB int8 per tile
constexpr int IX_A_COL = IX_TILE * 128;                // one 64-dim fp16 atom column, 16 KB
constexpr int IX_B_COL = 256 * 128;                    // B atom column for up to N = 256 rows
constexpr int IX_MAX_SEG = 1024;
constexpr int IX_OFF_A = 0;
constexpr int IX_OFF_B = IX_OFF_A + 2 * IX_A_COL;      // 32 KB
constexpr int IX_OFF_RAW = IX_OFF_B + 2 * IX_B_COL;    // 96 KB
constexpr int IX_OFF_BAR = IX_OFF_RAW + IX_STAGES * IX_RAW;
constexpr int IX_OFF_SEG = IX_OFF_BAR + 128;
constexpr int IX_SMEM = IX_OFF_SEG + IX_MAX_SEG * 16 + 4 * 64 * 4 + 2 * IX_MAX_SEG * 4 + 1024;

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

__global__ void __launch_bounds__(IX_THREADS, 1)
indexer_kernel(Dev D, int il, int n_tok, const int32_t* __restrict__ req_of, const int32_t* __restrict__ limit_of,
               const int8_t* __restrict__ qg, const int8_t* __restrict__ wg, int64_t* __restrict__ scores) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + IX_OFF_BAR);     // [0..S) full, [S] mma
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + IX_OFF_BAR + 8 * (IX_STAGES + 1));
  int32_t* s_nseg = reinterpret_cast<int32_t*>(tmem_slot + 1);
  int32_t* s_flag = s_nseg + 1;
  IxSeg* segs = reinterpret_cast<IxSeg*>(smem + IX_OFF_SEG);
  int32_t* s_w = reinterpret_cast<int32_t*>(smem + IX_OFF_SEG + IX_MAX_SEG * 16);   // [4][64]
  int32_t* s_req = s_w + 4 * 64;                                                      // [n_tok]
  int32_t* s_lim = s_req + IX_MAX_SEG;                                                // [n_tok]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hi = D.n_idx_heads;
  const int8_t* keys = D.idx[il];

  // ---- request segments of the batch (tokens of one request are contiguous) ----
  for (int t = tid; t < n_tok; t += IX_THREADS) {
    int r = req_of[t], lim = limit_of[t];
    if (r < 0 || r >= D.max_requests || lim < 0 || lim > D.max_ctx) {
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
    for (int st = 0; st <= IX_STAGES; ++st) mbar_init(smem_u32(&bars[st]), 1);
    fence_mbar_init();
    *s_flag = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 256);
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
  // issue the bulk copies of the (up to two) key pages of local item i into its stage
  auto issue = [&](int i) {
    int item = (int)blockIdx.x + i * (int)gridDim.x;
    int sg = seg_of(item);
    int tile = item - (sg ? segs[sg - 1].tile_end : 0);
    int r = s_req[segs[sg].first];
    int stage = i % IX_STAGES;
    uint32_t bar = smem_u32(&bars[stage]);
    uint32_t dst = smem_u32(smem + IX_OFF_RAW + stage * IX_RAW);
    int npg = ((tile * IX_TILE + PAGE) < segs[sg].maxlim) ? 2 : 1;
    int ip[2] = {-1, -1};
    uint32_t bytes = 0;
    for (int k = 0; k < npg; ++k) {
      int v = D.idx_bt[(size_t)r * D.max_pages + tile * 2 + k];
      if (v < 0 || v >= D.num_idx_pages) {
        set_status(D.status, HS_ERR_BAD_ID);
        continue;
      }
      ip[k] = v;
      bytes += IDX_PAGE_BYTES;
    }
    mbar_expect_tx(bar, bytes);
    for (int k = 0; k < 2; ++k)
      if (ip[k] >= 0) bulk_g2s(dst + k * IDX_PAGE_BYTES, keys + (size_t)ip[k] * IDX_PAGE_BYTES, IDX_PAGE_BYTES, bar);
  };

  int issued = 0;   // meaningful in thread 0 only
  if (tid == 0) {
    for (int i = 0; i < min(n_local, IX_STAGES); ++i) issue(i);
    issued = min(n_local, IX_STAGES);
  }

  int cur_seg = -1;
  bool dead = false;
  int died_at = 0;
  for (int i = 0; i < n_local && !dead; ++i) {
    const int item = (int)blockIdx.x + i * (int)gridDim.x;
    const int sg = seg_of(item);
    const IxSeg S = segs[sg];
    const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
    const int key0 = tile * IX_TILE;
    const int N = ((S.ntok * Hi) + 15) & ~15;

    if (sg != cur_seg) {
      // load the segment's queries as the B operand: row n = j * Hi + h, K-major SW128
      uint8_t* B = smem + IX_OFF_B;
      const int rows = N;
      for (int c = tid; c < rows * 8; c += IX_THREADS) {
        int row = c >> 3, ch16 = c & 7;            // 8 chunks of 16 int8 per 128-dim row
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < S.ntok * Hi) {
          int j = row / Hi, h = row - j * Hi;
          v = *reinterpret_cast<const uint4*>(qg + ((size_t)(S.first + j) * Hi + h) * IDX_DIM + ch16 * 16);
        }
        uint4 c0, c1;
        i8x16_to_f16(v, c0, c1);
        int dim0 = ch16 * 16;                       // 16 dims -> fp16 chunks (dim0/8, dim0/8+1)
        int col = dim0 >> 6;                        // atom column
        int chunk = (dim0 & 63) >> 3;
        uint8_t* base = B + col * IX_B_COL;
        *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk)) = c0;
        *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk + 1)) = c1;
      }
      for (int c = tid; c < 4 * 64; c += IX_THREADS) {
        int j = c >> 6, h = c & 63;
        int w = 0;
        if (j < S.ntok && h < Hi) {
          w = wg[(size_t)(S.first + j) * Hi + h];
          if (w < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); w = 0; }
        }
        s_w[c] = w;
      }
      cur_seg = sg;
    }

    // ---- wait for the key tile, widen to fp16 (A operand: M = keys, K-major) ----
    const int stage = i % IX_STAGES;
    if (!mbar_wait(smem_u32(&bars[stage]), (i / IX_STAGES) & 1, D.status)) *s_flag = 1;
    const uint8_t* raw = smem + IX_OFF_RAW + stage * IX_RAW;
    uint8_t* A = smem + IX_OFF_A;
    for (int c = tid; c < IX_TILE * 8; c += IX_THREADS) {
      int row = c >> 3, ch16 = c & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (key0 + row < S.maxlim) v = *reinterpret_cast<const uint4*>(raw + row * IDX_DIM + ch16 * 16);
      uint4 c0, c1;
      i8x16_to_f16(v, c0, c1);
      int dim0 = ch16 * 16;
      uint8_t* base = A + (dim0 >> 6) * IX_A_COL;
      int chunk = (dim0 & 63) >> 3;
      *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk)) = c0;
      *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk + 1)) = c1;
    }
    fence_proxy_async();
    __syncthreads();
    if (*s_flag) { dead = true; died_at = i; break; }
    if (tid == 0) {
      if (i + IX_STAGES < n_local) {
        issue(i + IX_STAGES);
        issued = i + IX_STAGES + 1;
      }
      tc_fence_after();
      const uint32_t idesc = idesc_f16(128, N, false, false);
      const uint32_t a0 = smem_u32(A), b0 = smem_u32(smem + IX_OFF_B);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * IX_A_COL + (kk & 3) * 32, 16, 1024);
        uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * IX_B_COL + (kk & 3) * 32, 16, 1024);
        umma_f16(tmem, ad, bd, idesc, kk > 0);
      }
      umma_commit(smem_u32(&bars[IX_STAGES]));
    }
    if (!mbar_wait(smem_u32(&bars[IX_STAGES]), i & 1, D.status)) *s_flag = 1;
    tc_fence_after();

    // ---- epilogue: warp w reads TMEM lanes 32*(w%4).., tokens j = w/4, w/4 + 2 ----
    {
      const int quad = warp & 3;
      const int key = key0 + quad * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
      for (int j = warp >> 2; j < 4; j += 2) {
        if (j >= S.ntok) break;      // warp-uniform
        const int lim = s_lim[S.first + j];
        long long acc = 0;
        for (int h0 = 0; h0 < Hi; h0 += 16) {
          uint32_t r[16];
          tmem_ld16(lane_addr + (uint32_t)(j * Hi + h0), r);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            int v = __float2int_rn(__uint_as_float(r[k]));
            v = max(v, 0);
            acc += (long long)v * s_w[j * 64 + h0 + k];
          }
        }
        if (key < lim) scores[(size_t)(S.first + j) * D.max_ctx + key] = acc;
      }
    }
    tc_fence_before();
    __syncthreads();
    if (*s_flag) { dead = true; died_at = i + 1; }
  }
  __syncthreads();
  if (dead && tid == 0) {
    // drain bulk copies still in flight before the CTA's shared memory goes away
    for (int k = died_at; k < issued; ++k) mbar_wait(smem_u32(&bars[k % IX_STAGES]), (k / IX_STAGES) & 1, D.status);
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ----------------------------------------------------------------------------------
// Select kernel
// ----------------------------------------------------------------------------------
constexpr int SEL_CL = 8;
constexpr int SEL_THREADS = 512;
constexpr int SEL_BINS = 4096;
constexpr int SEL_SLICE = SEL_BINS / SEL_CL;
constexpr int SEL_CACHE = 24576;                       // scores cached in shared memory per CTA
constexpr int SEL_SMEM = SEL_CACHE * 8 + 1024;

// monotone level-1 bucket: exact below 64, then 64 buckets per octave
__device__ __forceinline__ int bucket1(long long v) {
  if (v < 64) return v < 0 ? 0 : (int)v;
  int e = 63 - __clzll(v);
  int m = (int)((v >> (e - 6)) & 63);
  return 64 + (e - 6) * 64 + m;
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

__global__ void __cluster_dims__(SEL_CL, 1, 1) __launch_bounds__(SEL_THREADS, 1)
select_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
              int32_t* __restrict__ topk) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int tok = blockIdx.x / SEL_CL;
  const int K = D.topk;
  __shared__ uint32_t hist[SEL_BINS];
  __shared__ uint32_t tot[SEL_SLICE];
  __shared__ int warp_tot[32];
  __shared__ int s_sum;
  __shared__ long long s_above;
  __shared__ int s_bin;
  __shared__ int cnt[2];
  extern __shared__ __align__(16) uint8_t sel_dyn[];
  long long* cache = reinterpret_cast<long long*>(sel_dyn);

  int n = limit_of[tok];
  n = max(0, min(n, D.max_ctx));
  int32_t* out = topk + (size_t)tok * K;
  if (n <= K) {           // every earlier token is selected (uniform across the cluster)
    if (crank == 0)
      for (int i = threadIdx.x; i < K; i += blockDim.x) out[i] = i < n ? i : -1;
    return;
  }
  const long long* s = reinterpret_cast<const long long*>(scores) + (size_t)tok * ld;
  const int per = (n + SEL_CL - 1) / SEL_CL;
  const int lo = crank * per, hi = min(n, lo + per);
  const int cnt_local = max(0, hi - lo);
  const bool cached = per <= SEL_CACHE;

  int need = K;
  int level = 0;
  long long base = 0, width = 0;   // level >= 1: value range [base, base + width)
  int shift = 0;
  for (;; ++level) {
    for (int b = threadIdx.x; b < SEL_BINS; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < cnt_local; i += blockDim.x) {
      long long v;
      if (level == 0) {
        v = s[lo + i];
        if (cached) cache[i] = v;
        atomicAdd(&hist[bucket1(v)], 1u);
      } else {
        v = cached ? cache[i] : s[lo + i];
        if (v >= base && v - base < width) atomicAdd(&hist[(int)((v - base) >> shift)], 1u);
      }
    }
    cluster.sync();
    // reduce my slice of bins over the cluster
    for (int b = threadIdx.x; b < SEL_SLICE; b += blockDim.x) {
      uint32_t a = 0;
#pragma unroll
      for (int r = 0; r < SEL_CL; ++r) a += cluster.map_shared_rank(hist, r)[crank * SEL_SLICE + b];
      tot[b] = a;
    }
    cluster.sync();
    for (int b = threadIdx.x; b < SEL_BINS; b += blockDim.x)
      hist[b] = cluster.map_shared_rank(tot, b / SEL_SLICE)[b % SEL_SLICE];
    __syncthreads();
    // find the bin holding the need-th largest value, scanning from the top bin
    if (threadIdx.x == 0) { s_bin = 0; s_above = 0; }
    __syncthreads();
    {
      const int per_t = SEL_BINS / SEL_THREADS;     // 8 bins per thread, thread 0 = top bins
      int local = 0;
      for (int k = 0; k < per_t; ++k) local += hist[SEL_BINS - 1 - (threadIdx.x * per_t + k)];
      int before = block_excl_scan(local, warp_tot, nullptr);
      if (before < need && need <= before + local) {
        int cum = before;
        for (int k = 0; k < per_t; ++k) {
          int b = SEL_BINS - 1 - (threadIdx.x * per_t + k);
          if (cum + (int)hist[b] >= need) { s_bin = b; s_above = cum; break; }
          cum += hist[b];
        }
      }
      __syncthreads();
    }
    const int B = s_bin;
    need -= (int)s_above;
    if (level == 0) {
      if (B < 64) { base = B; width = 1; }
      else {
        int e = (B - 64) / 64 + 6, m = (B - 64) % 64;
        base = (1ll << e) + ((long long)m << (e - 6));
        width = 1ll << (e - 6);
      }
    } else {
      base += (long long)B << shift;
      width = 1ll << shift;
    }
    if (width == 1) break;
    int lw = 63 - __clzll(width);
    shift = lw > 12 ? lw - 12 : 0;
  }
  const long long tau = base;   // the K-th largest score; `need` of its ties are taken

  // ---- counts per CTA, prefix over the cluster (CTA ranks own ascending ranges) ----
  int gt = 0, eq = 0;
  for (int i = threadIdx.x; i < cnt_local; i += blockDim.x) {
    long long v = cached ? cache[i] : s[lo + i];
    gt += v > tau;
    eq += v == tau;
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (threadIdx.x == 0) { cnt[0] = 0; cnt[1] = 0; }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) { atomicAdd(&cnt[0], gt); atomicAdd(&cnt[1], eq); }
  cluster.sync();
  int out_off = 0, eq_before = 0;
  for (int r = 0; r < crank; ++r) {
    int* pc = cluster.map_shared_rank(cnt, r);
    int g = pc[0], e = pc[1];
    int take = max(0, min(e, need - eq_before));
    out_off += g + take;
    eq_before += e;
  }
  const int my_take = max(0, min(cnt[1], need - eq_before));
  // ---- ordered compaction of my range ----
  int eq_run = 0, sel_run = 0;
  constexpr int IPT = 4;
  for (int t0 = 0; t0 < cnt_local; t0 += SEL_THREADS * IPT) {
    int idx0 = t0 + threadIdx.x * IPT;
    long long v[IPT];
    int e_local = 0;
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      int i = idx0 + k;
      v[k] = (i < cnt_local) ? (cached ? cache[i] : s[lo + i]) : LLONG_MIN;
      e_local += v[k] == tau;
    }
    int e_tot;
    int e_before = block_excl_scan(e_local, warp_tot, &s_sum) + eq_run;
    e_tot = s_sum;
    int sflags = 0, s_local = 0;
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      bool sel = v[k] > tau;
      if (v[k] == tau) { sel = e_before < my_take; ++e_before; }
      sflags |= (sel ? 1 : 0) << k;
      s_local += sel;
    }
    int s_before = block_excl_scan(s_local, warp_tot, &s_sum) + sel_run;
    int s_tot = s_sum;
#pragma unroll
    for (int k = 0; k < IPT; ++k)
      if (sflags >> k & 1) {
        const int pos = out_off + s_before++;
        if (pos < K) out[pos] = lo + idx0 + k;
        else set_status(D.status, HS_ERR_BAD_ID);
      }
    eq_run += e_tot;
    sel_run += s_tot;
    __syncthreads();
  }
  cluster.sync();   // peers may still read cnt[] until here
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
  indexer_kernel<<<num_sms(), IX_THREADS, IX_SMEM, st>>>(p->d, il, n, d_req, d_limit, d_q, d_w, d_scores);
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

hs_status launch_select(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                        int32_t* d_topk, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_SMEM) !=
        cudaSuccess)
      return HS_ERR_CUDA;
    attr = true;
  }
  select_kernel<<<n * SEL_CL, SEL_THREADS, SEL_SMEM, st>>>(p->d, scores, ld, d_limit, d_topk);
  return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

}  // namespace hs
