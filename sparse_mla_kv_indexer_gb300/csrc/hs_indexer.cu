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
//  * key pages (64 x 128 B) arrive by bulk copy (TMA unit) into a ring of 6-12
//    stages (all shared memory the query operand leaves free), filled by a
//    producer warp that fetches page ids 32 tiles ahead; converter warps, an MMA warp and epilogue warps
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

#include <atomic>
#include <map>
#include <mutex>

#include "hs_select.cuh"

namespace cg = cooperative_groups;

namespace hs {

// ----------------------------------------------------------------------------------
// Scoring kernel
// ----------------------------------------------------------------------------------
// Warp roles (448 threads):
//   warps 0-7   epilogue, two warpgroups on alternate tiles (one tile's TMEM reads
//               and dependent arithmetic overlap the other's): TMEM accumulator ->
//               ReLU, head weights, int64 scores
//   warps 8-11  convert: raw int8 key tile -> fp16 A tile; queries -> fp16 B operand
//   warp 12     producer: bulk copies of key pages into the stage ring
//   warp 13     MMA issuer: tcgen05.mma into one of the TMEM accumulators
constexpr int IX_THREADS = 448;
constexpr int IX_EPI_GROUPS = 2;
constexpr int IX_CONV_WARP0 = 8;
constexpr int IX_CONV = 128;                           // converter threads
constexpr int IX_PRODUCER_WARP = 12, IX_MMA_WARP = 13;
constexpr int IX_MAX_A = 4;                            // fp16 A tiles in flight
constexpr int IX_MAX_STAGES = 12;
constexpr int IX_TILE = 128;
constexpr int IX_RAW = IX_TILE * IDX_DIM;              // 16 KB int8 per tile
constexpr int IX_A_COL = IX_TILE * 128;                // one 64-dim fp16 atom column, 16 KB
constexpr int IX_A = 2 * IX_A_COL;                     // 32 KB per A tile
constexpr int IX_SMEM_BUDGET = 227 * 1024;
constexpr int IX_TMEM_COLS = 512;                      // accumulators: 2 x 256 .. 8 x 64 columns
constexpr int IX_MAX_ACC = 8;

// Shared-memory layout of one launch, sized by the batch geometry so the key
// ring gets every byte the query operand does not need.
struct IxLayout {
  int n_a;        // fp16 A tiles (3 or 4: conversion runs ahead of the MMA)
  int b_col;      // bytes per 64-dim atom column of the query operand (n_max rows x 128 B)
  int off_b, off_raw, off_bar, off_seg, off_hist, stages, smem;   // off_hist: 0 = no histogram
  int acc_cols;   // TMEM columns per accumulator (power of two >= n_max rows)
  int n_acc;      // accumulators in flight between the MMA warp and the epilogue
};

IxLayout ix_layout(int n_max_rows, int max_tokens, bool hist) {
  IxLayout L;
  L.b_col = n_max_rows * 128;
  const int hist_bytes = hist ? SEL_BINS * 4 : 0;
  const int tail = 512 + max_tokens * 16 + IX_EPI_GROUPS * (4 * 64 * 4 + 64) + 2 * max_tokens * 4 + hist_bytes + 1024;
  // as many A tiles as leave at least three key stages, then every remaining byte to the key ring
  for (L.n_a = IX_MAX_A; L.n_a > 2; --L.n_a)
    if ((IX_SMEM_BUDGET - L.n_a * IX_A - 2 * L.b_col - tail) / IX_RAW >= 3) break;
  L.off_b = L.n_a * IX_A;
  L.off_raw = L.off_b + 2 * L.b_col;
  int stages = (IX_SMEM_BUDGET - L.off_raw - tail) / IX_RAW;
  L.stages = stages > IX_MAX_STAGES ? IX_MAX_STAGES : stages;
  L.off_bar = L.off_raw + L.stages * IX_RAW;
  L.off_seg = L.off_bar + 512;
  L.off_hist = hist ? L.off_seg + max_tokens * 16 + IX_EPI_GROUPS * (4 * 64 * 4 + 64) + 2 * max_tokens * 4 : 0;
  L.smem = L.off_seg + max_tokens * 16 + IX_EPI_GROUPS * (4 * 64 * 4 + 64) + 2 * max_tokens * 4 + hist_bytes + 1024;
  L.acc_cols = 32;
  while (L.acc_cols < n_max_rows) L.acc_cols <<= 1;
  L.n_acc = IX_TMEM_COLS / L.acc_cols < IX_MAX_ACC ? IX_TMEM_COLS / L.acc_cols : IX_MAX_ACC;
  return L;
}

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
// Named barrier over n threads that also ORs a flag across them: every thread
// leaves with the same answer.
__device__ __forceinline__ int named_sync_or(int id, int n, int flag) {
  int out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}"
      : "=r"(out) : "r"(flag), "r"(id), "r"(n) : "memory");
  return out;
}

__global__ void __launch_bounds__(IX_THREADS, 1)
indexer_kernel(Dev D, int il, int n_tok, const int32_t* __restrict__ req_of, const int32_t* __restrict__ limit_of,
               const int8_t* __restrict__ qg, const int8_t* __restrict__ wg, int64_t* __restrict__ scores,
               int ld, IxLayout L, uint32_t* __restrict__ hist0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NS = L.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* raw_full = bars;                      // [NS]
  uint64_t* raw_empty = bars + IX_MAX_STAGES;     // [NS]
  uint64_t* a_full = bars + 2 * IX_MAX_STAGES;    // [n_a]
  uint64_t* a_empty = a_full + IX_MAX_A;          // [n_a]
  uint64_t* t_full = a_empty + IX_MAX_A;          // [n_acc]
  uint64_t* t_empty = t_full + IX_MAX_ACC;        // [n_acc]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(t_empty + IX_MAX_ACC);
  int32_t* s_nseg = reinterpret_cast<int32_t*>(tmem_slot + 1);
  int32_t* s_dead = s_nseg + 1;
  int32_t* s_issued = s_nseg + 2;
  int32_t* s_consumed = s_nseg + 3;
  IxSeg* segs = reinterpret_cast<IxSeg*>(smem + L.off_seg);
  int32_t* s_w = reinterpret_cast<int32_t*>(segs + D.max_tokens);   // [IX_EPI_GROUPS][4][64], per warpgroup
  int32_t* s_req = s_w + IX_EPI_GROUPS * 4 * 64;                     // [n_tok]
  int32_t* s_lim = s_req + D.max_tokens;                             // [n_tok]
  int32_t* s_wsum = s_lim + D.max_tokens;                            // [IX_EPI_GROUPS][4][4], per warpgroup
  // hist0 (one query token, wide selection): the selection's level-0 histogram of
  // this CTA's scores, added to the selection's global sums at the end
  uint32_t* s_hist = hist0 ? reinterpret_cast<uint32_t*>(smem + L.off_hist) : nullptr;   // [SEL_BINS]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hi = D.n_idx_heads;
  const int8_t* keys = D.idx[il];

  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), IX_TMEM_COLS);
  if (tid == 0) {
    for (int b = 0; b < 2 * IX_MAX_STAGES + 2 * IX_MAX_A + 2 * IX_MAX_ACC; ++b) mbar_init(smem_u32(&bars[b]), 1);
    fence_mbar_init();
  }
  if (s_hist)
    for (int b = tid; b < SEL_BINS; b += IX_THREADS) s_hist[b] = 0;
  // Request ids, limits, queries, weights and the index block table are inputs,
  // final before the preceding kernel started: the segments, page ids, query operand
  // and weights are set up while it finishes. The producer waits for that kernel
  // before its first key copy (the keys may have been appended by it); the score and
  // histogram writes follow the copies.
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
    *s_dead = 0;
    *s_issued = 0;
    *s_consumed = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nseg = *s_nseg;
  const int total = nseg ? segs[nseg - 1].tile_end : 0;
  // With several requests each CTA takes a contiguous run of tiles: a CTA then meets
  // one or two request boundaries in the whole launch, and each boundary drains its
  // pipeline (the query operand and the head weights of the next request are loaded
  // once the previous request's MMAs and epilogues are done). A single request is
  // dealt round robin, which measured faster (the CTAs sweep the keys together).
  const bool runs = nseg > 1;
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int first_item = runs ? (int)blockIdx.x * per : (int)blockIdx.x;
  const int n_local = runs ? (total > first_item ? min(per, total - first_item) : 0)
                           : (total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0);

  auto seg_of = [&](int item) {
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (segs[mid].tile_end > item) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  auto item_of = [&](int i) { return runs ? first_item + i : first_item + i * (int)gridDim.x; };

  if (warp == IX_PRODUCER_WARP) {
    // ------------------------------ producer ------------------------------
    // Lane l holds the key-page ids of tile (32c + l) of the current chunk c and
    // of the next chunk, so no copy waits on a dependent page-table load.
    auto fetch = [&](int i, int& p0, int& p1) {
      p0 = p1 = -2;
      if (i < n_local) {
        const int item = item_of(i);
        const int sg = seg_of(item);
        const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
        const int32_t* bt = D.idx_bt + (size_t)s_req[segs[sg].first] * D.max_pages + tile * 2;
        p0 = bt[0];
        p1 = ((tile * IX_TILE + PAGE) < segs[sg].maxlim) ? bt[1] : -2;   // -2: page beyond the limit
      }
    };
    int c0, c1, n0, n1;
    fetch(lane, c0, c1);
    fetch(32 + lane, n0, n1);
    griddep_wait();
    griddep_launch();
    for (int i = 0; i < n_local; ++i) {
      if (i > 0 && (i & 31) == 0) {
        c0 = n0;
        c1 = n1;
        fetch(i + 32 + lane, n0, n1);
      }
      const int ip0 = __shfl_sync(0xffffffffu, c0, i & 31);
      const int ip1 = __shfl_sync(0xffffffffu, c1, i & 31);
      int dead = 0;
      if (lane == 0) {
        const int rs = i % NS;
        if (i >= NS && !mbar_wait(smem_u32(&raw_empty[rs]), ((i / NS) - 1) & 1, D.status)) *s_dead = 1;
        dead = *(volatile int32_t*)s_dead;
        if (!dead) {
          const uint32_t bar = smem_u32(&raw_full[rs]);
          const uint32_t dst = smem_u32(smem + L.off_raw + rs * IX_RAW);
          const int ips[2] = {ip0, ip1};
          uint32_t bytes = 0;
          for (int k = 0; k < 2; ++k) {
            if (ips[k] == -2) continue;
            if (ips[k] < 0 || ips[k] >= D.num_idx_pages) { set_status(D.status, HS_ERR_BAD_ID); continue; }
            bytes += IDX_PAGE_BYTES;
          }
          mbar_expect_tx(bar, bytes);
          for (int k = 0; k < 2; ++k)
            if (ips[k] >= 0 && ips[k] < D.num_idx_pages)
              bulk_g2s(dst + k * IDX_PAGE_BYTES, keys + (size_t)ips[k] * IDX_PAGE_BYTES, IDX_PAGE_BYTES, bar);
          *s_issued = i + 1;
        }
      }
      if (__shfl_sync(0xffffffffu, dead, 0)) break;
    }
  } else if (warp == IX_MMA_WARP) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      for (int i = 0; i < n_local; ++i) {
        const int ab = i % L.n_a, tb = i % L.n_acc;
        if (!mbar_wait(smem_u32(&a_full[ab]), (i / L.n_a) & 1, D.status)) { *s_dead = 1; break; }
        if (i >= L.n_acc && !mbar_wait(smem_u32(&t_empty[tb]), ((i / L.n_acc) - 1) & 1, D.status)) {
          *s_dead = 1;
          break;
        }
        if (*(volatile int32_t*)s_dead) break;
        tc_fence_after();
        const IxSeg S = segs[seg_of(item_of(i))];
        const int N = ((S.ntok * Hi) + 15) & ~15;
        const uint32_t idesc = idesc_f16(128, N, false, false);
        const uint32_t a0 = smem_u32(smem + ab * IX_A), b0 = smem_u32(smem + L.off_b);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * IX_A_COL + (kk & 3) * 32, 16, 1024);
          uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * L.b_col + (kk & 3) * 32, 16, 1024);
          umma_f16(tmem + tb * L.acc_cols, ad, bd, idesc, kk > 0);
        }
        umma_commit(smem_u32(&a_empty[ab]));
        umma_commit(smem_u32(&t_full[tb]));
      }
    }
  } else if (warp >= IX_CONV_WARP0) {
    // ------------------------------ converters ------------------------------
    const int ct = tid - IX_CONV_WARP0 * 32;
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
        if (i > 0) ok = mbar_wait(smem_u32(&a_empty[(i - 1) % L.n_a]), ((i - 1) / L.n_a) & 1, D.status);
        uint8_t* B = smem + L.off_b;
        const int N = ((S.ntok * Hi) + 15) & ~15;
        for (int c = ct; c < N * 8; c += IX_CONV) {
          const int row = c >> 3, ch16 = c & 7;       // 8 chunks of 16 int8 per 128-dim row
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < S.ntok * Hi) {
            const int j = row / Hi, h = row - j * Hi;
            v = *reinterpret_cast<const uint4*>(qg + ((size_t)(S.first + j) * Hi + h) * IDX_DIM + ch16 * 16);
          }
          uint4 c0, c1;
          i8x16_to_f16(v, c0, c1);
          const int dim0 = ch16 * 16;
          uint8_t* base = B + (dim0 >> 6) * L.b_col;
          const int chunk = (dim0 & 63) >> 3;
          *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk)) = c0;
          *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk + 1)) = c1;
        }
        cur_seg = sg;
      }
      const int rs = i % NS, ab = i % L.n_a;
      if (ok) ok = mbar_wait(smem_u32(&raw_full[rs]), (i / NS) & 1, D.status);
      if (ok && i >= L.n_a) ok = mbar_wait(smem_u32(&a_empty[ab]), ((i / L.n_a) - 1) & 1, D.status);
      if (!ok) *s_dead = 1;
      const uint8_t* raw = smem + L.off_raw + rs * IX_RAW;
      uint8_t* A = smem + ab * IX_A;
      // chunk c -> (row, 16-byte piece): each group of 8 lanes takes pieces 0-3 of one
      // row and pieces 4-7 of its neighbour, so its loads cover all 32 banks once and
      // its two swizzled stores land on 8 distinct 16-byte slots (no bank conflicts)
      auto piece_of = [](int c, int& row, int& ch16) {
        const int half = (c >> 2) & 1;
        row = 2 * (c >> 4) + (((c >> 3) & 1) ^ half);
        ch16 = half * 4 + (c & 3);
      };
      constexpr int CPT = IX_TILE * 8 / IX_CONV;   // 16-byte chunks per converter thread
      uint4 v[CPT];
#pragma unroll
      for (int k = 0; k < CPT; ++k) {   // all loads first
        int row, ch16;
        piece_of(ct + k * IX_CONV, row, ch16);
        v[k] = key0 + row < S.maxlim ? *reinterpret_cast<const uint4*>(raw + row * IDX_DIM + ch16 * 16)
                                     : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        int row, ch16;
        piece_of(ct + k * IX_CONV, row, ch16);
        uint4 c0, c1;
        i8x16_to_f16(v[k], c0, c1);
        const int dim0 = ch16 * 16;
        uint8_t* base = A + (dim0 >> 6) * IX_A_COL;
        const int chunk = (dim0 & 63) >> 3;
        *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk)) = c0;
        *reinterpret_cast<uint4*>(base + sw128_chunk(row, chunk + 1)) = c1;
      }
      fence_proxy_async();
      named_sync(1, IX_CONV);
      if (ct == 0) {
        *s_consumed = i + 1;
        mbar_arrive(smem_u32(&raw_empty[rs]));
        mbar_arrive(smem_u32(&a_full[ab]));
      }
      if (*(volatile int32_t*)s_dead) break;
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    // warpgroup grp takes tiles i = grp, grp + 2, ...; the accumulator count is even,
    // so each accumulator stays with one warpgroup and its phase waits never alias
    const int grp = warp >> 2, et = tid & 127;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int32_t* sw = s_w + grp * 4 * 64;
    int32_t* swsum = s_wsum + grp * 16;
    int cur_seg = -1;
    for (int i = grp; i < n_local; i += IX_EPI_GROUPS) {
      const int item = item_of(i);
      const int sg = seg_of(item);
      const IxSeg S = segs[sg];
      const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
      const int key = tile * IX_TILE + et;
      if (sg != cur_seg) {
        named_sync(2 + grp, 128);
        for (int c = et; c < 4 * 64; c += 128) {
          const int j = c >> 6, h = c & 63;
          int w = 0;
          if (j < S.ntok && h < Hi) {
            w = wg[(size_t)(S.first + j) * Hi + h];
            if (w < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); w = 0; }
          }
          sw[c] = w;
        }
        named_sync(2 + grp, 128);
        if (et < 16) {   // sum of the weights of each 16-head group, per token
          int t = 0;
          for (int k = 0; k < 16; ++k) t += sw[(et >> 2) * 64 + (et & 3) * 16 + k];
          swsum[et] = t;
        }
        named_sync(2 + grp, 128);
        cur_seg = sg;
      }
      const int tb = i % L.n_acc;
      // a failed wait is recorded and the tile run through without stores, so that the
      // warpgroup's decision to stop is taken together at the barrier below
      const int ok = mbar_wait(smem_u32(&t_full[tb]), (i / L.n_acc) & 1, D.status);
      if (!ok) *s_dead = 1;
      tc_fence_after();
      // Exact integer epilogue without float->int conversions: every dot product
      // is an integer |d| <= 2^21 held exactly in fp32, so max(d, 0) + 2^23 has the
      // bit pattern 0x4B000000 + relu(d). With w <= 127, each w * relu(d) < 2^28 and
      // 16 of them sum below 2^32: 16 heads accumulate bits * w in uint32 (mod 2^32,
      // in four independent partial sums) and the offset 0x4B000000 * sum(w) comes
      // off once per group, which leaves the exact group sum; the groups add in 64 bits.
      for (int j = 0; j < S.ntok; ++j) {
        const int lim = s_lim[S.first + j];
        const uint32_t col0 = lane_base + (uint32_t)(tb * L.acc_cols + j * Hi);
        uint32_t r[64];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q * 16 < Hi) tmem_ld16(col0 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(r + q * 16));
        tmem_wait_ld();
        unsigned long long acc = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q * 16 < Hi) {
            uint32_t p[4] = {0u - 0x4B000000u * (uint32_t)swsum[j * 4 + q], 0u, 0u, 0u};
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int4 w4 = *reinterpret_cast<const int4*>(sw + j * 64 + q * 16 + k4 * 4);
              const int w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float d = fmaxf(__uint_as_float(r[q * 16 + k4 * 4 + k]), 0.f);
                p[k] += __float_as_uint(d + 8388608.f) * (uint32_t)w[k];
              }
            }
            acc += (uint32_t)((p[0] + p[1]) + (p[2] + p[3]));
          }
        }
        if (ok && key < lim) {
          scores[(size_t)(S.first + j) * ld + key] = (long long)acc;
          if (s_hist) atomicAdd(&s_hist[bucket1(sel_key((long long)acc, key))], 1u);
        }
      }
      tc_fence_before();
      if (named_sync_or(2 + grp, 128, *(volatile int32_t*)s_dead)) break;
      if (et == 0) mbar_arrive(smem_u32(&t_empty[tb]));
    }
    if (s_hist) {   // both warpgroups are done: this CTA's histogram to the global sums
      named_sync(4, IX_EPI_GROUPS * 128);
      for (int b = tid; b < SEL_BINS; b += IX_EPI_GROUPS * 128)
        if (s_hist[b]) atomicAdd(&hist0[b], s_hist[b]);
    }
  }
  __syncthreads();
  if (*s_dead && tid == IX_PRODUCER_WARP * 32) {
    // drain bulk copies still in flight before the CTA's shared memory goes away
    for (int k = *s_consumed; k < *s_issued; ++k)
      mbar_wait(smem_u32(&raw_full[k % NS]), (k / NS) & 1, D.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, IX_TMEM_COLS);
}

// ----------------------------------------------------------------------------------
// Select kernel (one cluster per query token); keys as in hs_select.cuh
// ----------------------------------------------------------------------------------
constexpr int SEL_THREADS = 512;
constexpr int SEL_CACHE = 12288;                       // keys cached in shared memory per CTA
constexpr int SEL_CAND = 2048;                         // candidates per CTA on the fast path
constexpr int SEL_LEAD = 4096;                         // candidates the cluster leader sorts
constexpr int SEL_PIECE = 2048;                       // keys per bulk copy of the streaming pass
constexpr int SEL_RING = 3;                            // pieces in flight
constexpr int SEL_STREAM_MAX = 81920;                  // keys per CTA whose buckets fit in shared memory
static_assert(16 * SEL_STREAM_MAX == HS_MAX_CTX, "the longest context fits the streaming pass");
// two layouts of the dynamic shared memory, chosen per launch by the chunk size:
//  cached    [keys SEL_CACHE x 8 B][lead][cand][buckets SEL_CACHE x 2 B]
//  streaming [buckets SEL_STREAM_MAX x 2 B][ring SEL_RING pieces; after pass 1: lead, cand]
constexpr int SEL_SMEM_CACHED = SEL_CACHE * 8 + SEL_CACHE * 2 + SEL_LEAD * 8 + SEL_CAND * 8;
constexpr int SEL_SMEM_STREAM = SEL_STREAM_MAX * 2 + SEL_RING * SEL_PIECE * 8;
constexpr int SEL_SMEM = (SEL_SMEM_CACHED > SEL_SMEM_STREAM ? SEL_SMEM_CACHED : SEL_SMEM_STREAM) + 16;
static_assert(SEL_LEAD * 8 + SEL_CAND * 8 <= SEL_RING * SEL_PIECE * 8, "lead and cand fit in the ring");

// shared-memory histogram increment (scores spread over many buckets, so plain
// atomics rarely collide within a warp)
__device__ __forceinline__ void hist_add(uint32_t* hist, int bin) { atomicAdd(&hist[bin], 1u); }

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

template <int CL>
__global__ void __launch_bounds__(SEL_THREADS, 1)
select_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
              int32_t* __restrict__ topk, int fp_keys) {
  uint32_t crank_u;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank_u));
  const int crank = (int)crank_u;
  constexpr int slice = SEL_BINS / CL;
  const int tok = blockIdx.x / CL;
  const int K = D.topk;
  const int tid = threadIdx.x;
  __shared__ uint32_t hist[SEL_BINS];      // level histograms (own partial, then cluster totals)
  __shared__ uint32_t tot[slice];          // cluster totals of this CTA's slice of bins
  __shared__ int warp_tot[32];
  __shared__ int s_bin, s_ncand, s_over, s_nsel, s_off, s_total_c, s_any_over;
  __shared__ int s_cnt[CL];
  __shared__ long long s_above;
  __shared__ unsigned long long s_tau;
  __shared__ __align__(8) uint64_t s_bar[SEL_RING];
  extern __shared__ __align__(16) uint8_t sel_dyn[];

  griddep_wait();
  griddep_launch();
  int n = limit_of[tok];
  n = max(0, min(n, D.max_ctx));
  int32_t* out = topk + (size_t)tok * K;
  if (n <= K) {           // every earlier token is selected (uniform across the cluster)
    if (crank == 0)
      for (int i = tid; i < K; i += blockDim.x) out[i] = i < n ? i : -1;
    return;
  }
  const long long* s = reinterpret_cast<const long long*>(scores) + (size_t)tok * ld;
  const int per = ((n + CL - 1) / CL + 1) & ~1;   // even, so every chunk starts 16-byte aligned
  const int lo = min(n, crank * per), hi = min(n, lo + per);
  const int cnt_local = max(0, hi - lo);
  // cached: the chunk's keys stay in shared memory; streaming (longer chunks, up to
  // SEL_STREAM_MAX since max_ctx <= HS_MAX_CTX): only their buckets do, and keys of
  // the threshold bucket are re-read from L2
  const bool cached = per <= SEL_CACHE;
  unsigned long long* cache = reinterpret_cast<unsigned long long*>(sel_dyn);             // cached: [SEL_CACHE]
  unsigned long long* lead = cached ? cache + SEL_CACHE                                    // [SEL_LEAD]
                                    : reinterpret_cast<unsigned long long*>(sel_dyn + SEL_STREAM_MAX * 2);
  unsigned long long* cand = lead + SEL_LEAD;                                              // [SEL_CAND]
  unsigned long long* ring = lead;                                                         // streaming pass 1
  uint16_t* bk = cached ? reinterpret_cast<uint16_t*>(cand + SEL_CAND)                    // [chunk] buckets
                        : reinterpret_cast<uint16_t*>(sel_dyn);
  int32_t* elist = reinterpret_cast<int32_t*>(lead);                                       // [K] after tau
  auto key_at = [&](int i) -> unsigned long long {
    if (cached) return cache[i];
    long long v = s[lo + i];
    return ((unsigned long long)max(v, 0ll) << 21) | (IDX_MASK - (unsigned long long)(lo + i));
  };

  // ---- level 0: histogram of bucket1(key); find the bucket of the K-th largest ----
  for (int b = tid; b < SEL_BINS; b += blockDim.x) hist[b] = 0;
  if (tid == 0) {
    s_ncand = 0; s_over = 0; s_bin = 0; s_above = 0;
    {
      for (int r = 0; r < SEL_RING; ++r) mbar_init(smem_u32(&s_bar[r]), 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (cached) {
    // the whole chunk arrives by bulk copy (TMA unit) in one round trip
    const int even = cnt_local & ~1;
    if (tid == 0) {
      const uint32_t bar = smem_u32(&s_bar[0]);
      mbar_expect_tx(bar, (uint32_t)even * 8u);
      for (int off = 0; off < even; off += 4096)
        bulk_g2s(smem_u32(cache + off), s + lo + off, (uint32_t)min(4096, even - off) * 8u, bar);
    }
    if (tid == 0 && (cnt_local & 1)) cache[cnt_local - 1] = (unsigned long long)s[lo + cnt_local - 1];
    if (!mbar_wait(smem_u32(&s_bar[0]), 0, D.status)) { /* recorded; the data below is then unreliable */ }
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < cnt_local; i += blockDim.x) {
      long long v = (long long)cache[i];
      if (v < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); v = 0; }
      const unsigned long long k = ((unsigned long long)v << 21) | (IDX_MASK - (unsigned long long)(lo + i));
      cache[i] = k;
      const int b = bucket_of(k, fp_keys);
      bk[i] = (uint16_t)b;
      hist_add(hist, b);
    }
  } else {
    // pieces of SEL_PIECE scores stream through a ring of bulk copies; each key's
    // bucket is kept, the key itself is not
    const int even = cnt_local & ~1;
    const int n_pieces = (even + SEL_PIECE - 1) / SEL_PIECE;
    auto issue = [&](int pc) {
      const int off = pc * SEL_PIECE, cnt = min(SEL_PIECE, even - off);
      const uint32_t bar = smem_u32(&s_bar[pc % SEL_RING]);
      mbar_expect_tx(bar, (uint32_t)cnt * 8u);
      bulk_g2s(smem_u32(ring + (pc % SEL_RING) * SEL_PIECE), s + lo + off, (uint32_t)cnt * 8u, bar);
    };
    if (tid == 0)
      for (int pc = 0; pc < SEL_RING && pc < n_pieces; ++pc) issue(pc);
    for (int pc = 0; pc < n_pieces; ++pc) {
      const bool ok = mbar_wait(smem_u32(&s_bar[pc % SEL_RING]), (pc / SEL_RING) & 1, D.status);
      if (__syncthreads_or(!ok)) break;   // a timeout (recorded) ends the pass for every thread
      const unsigned long long* piece = ring + (pc % SEL_RING) * SEL_PIECE;
      const int off = pc * SEL_PIECE, cnt = min(SEL_PIECE, even - off);
#pragma unroll 4
      for (int i = tid; i < cnt; i += blockDim.x) {
        long long v = (long long)piece[i];
        if (v < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); v = 0; }
        const int b = bucket_of(((unsigned long long)v << 21) | (IDX_MASK - (unsigned long long)(lo + off + i)), fp_keys);
        bk[off + i] = (uint16_t)b;
        hist_add(hist, b);
      }
      __syncthreads();   // the stage is read; it may be refilled
      if (tid == 0 && pc + SEL_RING < n_pieces) {
        fence_proxy_async();
        issue(pc + SEL_RING);
      }
    }
    if (tid == 0 && (cnt_local & 1)) {
      long long v = s[lo + cnt_local - 1];
      if (v < 0) { set_status(D.status, HS_ERR_BAD_WEIGHT); v = 0; }
      const int b = bucket_of(((unsigned long long)v << 21) | (IDX_MASK - (unsigned long long)(lo + cnt_local - 1)),
                              fp_keys);
      bk[cnt_local - 1] = (uint16_t)b;
      hist_add(hist, b);
    }
    __syncthreads();
  }
  int need = K;
  auto cluster_find = [&](void) {
    cluster_sync();
    for (int b = tid; b < slice; b += blockDim.x) {
      uint32_t part[CL];
#pragma unroll
      for (int r = 0; r < CL; ++r) part[r] = ld_cluster_u32(mapa(smem_u32(hist + crank * slice + b), r));
      uint32_t a = 0;
#pragma unroll
      for (int r = 0; r < CL; ++r) a += part[r];
      tot[b] = a;
    }
    cluster_sync();
    constexpr int PER = SEL_BINS / SEL_THREADS;   // 8 bins per thread
    uint32_t t[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int b = tid + k * SEL_THREADS;
      t[k] = ld_cluster_u32(mapa(smem_u32(tot + b % slice), b / slice));
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) hist[tid + k * SEL_THREADS] = t[k];
    if (tid == 0) { s_bin = 0; s_above = 0; }
    __syncthreads();
    int local = 0;
    for (int k = 0; k < PER; ++k) local += hist[SEL_BINS - 1 - (tid * PER + k)];
    int before = block_excl_scan(local, warp_tot, nullptr);
    if (before < need && need <= before + local) {
      int cum = before;
      for (int k = 0; k < PER; ++k) {
        int b = SEL_BINS - 1 - (tid * PER + k);
        if (cum + (int)hist[b] >= need) { s_bin = b; s_above = cum; break; }
        cum += hist[b];
      }
    }
    __syncthreads();
  };
  cluster_find();
  const int B0 = s_bin;
  need -= (int)s_above;

  // ---- fast path: collect the keys of bucket B0, the leader sorts them ----
#pragma unroll 4
  for (int i = tid; i < cnt_local; i += blockDim.x) {
    if (bk[i] == B0) {
      const unsigned long long k = key_at(i);
      int at = atomicAdd(&s_ncand, 1);
      if (at < SEL_CAND) cand[at] = k; else s_over = 1;
    }
  }
  cluster_sync();
  if (tid < 32) {
    int c = 0, o = 0;
    if (tid < CL) {
      c = (int)ld_cluster_u32(mapa(smem_u32(&s_ncand), tid));
      o = (int)ld_cluster_u32(mapa(smem_u32(&s_over), tid));
      s_cnt[tid] = c;
    }
    const int tc = __reduce_add_sync(0xffffffffu, min(c, SEL_CAND + 1));
    const int to = __reduce_or_sync(0xffffffffu, o);
    if (tid == 0) { s_total_c = tc; s_any_over = to; }
  }
  __syncthreads();
  const int total_c = s_total_c;
  const bool fast = !s_any_over && total_c <= SEL_LEAD;
  unsigned long long tau;
  if (fast) {
    if (crank == 0) {
      int np = 1;
      while (np < total_c) np <<= 1;
      // warp r copies peer r's candidates
      const int warp = tid >> 5, lane = tid & 31;
      if (warp < CL) {
        int base = 0;
        for (int r = 0; r < warp; ++r) base += s_cnt[r];
        const uint32_t pc = mapa(smem_u32(cand), warp);
        for (int i = lane; i < s_cnt[warp]; i += 32) lead[base + i] = ld_cluster_u64(pc + 8u * i);
      }
      for (int i = total_c + tid; i < np; i += blockDim.x) lead[i] = 0ull;
      __syncthreads();
      bitonic_desc(lead, np);
      if (tid == 0) s_tau = lead[need - 1];
    }
    cluster_sync();
    tau = ld_cluster_u64(mapa(smem_u32(&s_tau), 0));
  } else {
    // ---- slow path (crowded bucket): refine the key range level by level ----
    unsigned long long base, width;
    bucket_range(B0, fp_keys, base, width);
    while (width > 1) {
      const int shift = refine_shift(width);
      cluster_sync();     // peers finished reading tot[] of the previous level
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
    }
    tau = base;   // identical in every CTA of the cluster
  }

  // ---- emit: this CTA's selected tokens in ascending order, then place them ----
  // warp w owns a contiguous range of the chunk; one prefix over warp counts
  // orders the warps, ballots order the lanes.
  const int lane = tid & 31, wid = tid >> 5;
  constexpr int NW = SEL_THREADS / 32;
  const int wper = (cnt_local + NW - 1) / NW;
  const int wlo = min(cnt_local, wid * wper), whi = min(cnt_local, wlo + wper);
  // a key is selected when its bucket is above B0, or it is in B0 and not below tau
  auto selected = [&](int i) -> bool {
    const int b = bk[i];
    return b > B0 || (b == B0 && key_at(i) >= tau);
  };
  int wcount = 0;
#pragma unroll 4
  for (int i = wlo + lane; i < whi; i += 32) wcount += selected(i);
  wcount = __reduce_add_sync(0xffffffffu, wcount);
  if (lane == 0) warp_tot[wid] = wcount;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < wid; ++w) wbase += warp_tot[w];
  int sel_run = 0;
  for (int w = 0; w < NW; ++w) sel_run += warp_tot[w];
  for (int i0 = wlo; i0 < whi; i0 += 32) {
    const int i = i0 + lane;
    const bool sel = i < whi && selected(i);
    const unsigned m = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int pos = wbase + __popc(m & ((1u << lane) - 1));
      if (pos < K) elist[pos] = lo + i;
    }
    wbase += __popc(m);
  }
  __syncthreads();
  if (tid == 0) s_nsel = sel_run;
  cluster_sync();
  if (tid < 32) {
    const int c = (tid < crank) ? (int)ld_cluster_u32(mapa(smem_u32(&s_nsel), tid)) : 0;
    const int off = __reduce_add_sync(0xffffffffu, c);
    if (tid == 0) s_off = off;
  }
  __syncthreads();
  const int off = s_off;
  for (int i = tid; i < sel_run; i += blockDim.x) {
    if (off + i < K && i < K) out[off + i] = elist[i];
    else set_status(D.status, HS_ERR_BAD_ID);
  }
  cluster_sync();   // peers may still read this CTA's shared memory until here
}

int num_sms() {   // of the current device, looked up once per device
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDev) dev = 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

hs_status ensure_kernel_attrs(const void* kernel, int smem, bool nonportable_cluster) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;   // (kernel, device) -> limit set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  const auto it = done.find(key);
  if (it != done.end() && it->second >= smem) return HS_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      (nonportable_cluster && cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                                  cudaSuccess)) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  done[key] = smem;
  return HS_OK;
}

hs_status launch_indexer(hs_pool* p, int il, int n, const int32_t* d_req, const int32_t* d_limit,
                         const int8_t* d_q, const int8_t* d_w, int64_t* d_scores, uint32_t* d_hist0,
                         cudaStream_t st) {
  const int n_max = ((p->cfg.max_q_per_req * p->cfg.n_idx_heads) + 15) & ~15;
  const IxLayout L = ix_layout(n_max, p->cfg.max_tokens, d_hist0 != nullptr);
  if (L.stages < 2) return HS_ERR_INVALID;
  if (ensure_kernel_attrs(indexer_kernel, L.smem) != HS_OK) return HS_ERR_CUDA;
  return launch_pdl(indexer_kernel, dim3(num_sms()), dim3(IX_THREADS), L.smem, st, 0, p->d, il, n, d_req, d_limit,
                    d_q, d_w, d_scores, p->cfg.max_ctx, L, d_hist0);
}

template <int CL>
hs_status launch_select_cl(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                           int32_t* d_topk, bool fp_keys, cudaStream_t st) {
  if (ensure_kernel_attrs(select_kernel<CL>, SEL_SMEM, CL > 8) != HS_OK) return HS_ERR_CUDA;
  return launch_pdl(select_kernel<CL>, dim3(n * CL), dim3(SEL_THREADS), SEL_SMEM, st, CL, p->d, scores, ld, d_limit,
                    d_topk, fp_keys ? 1 : 0);
}

int select_wide_groups(hs_pool* p, int n, bool wide_ok) {
  // few query tokens: one wide group of co-resident CTAs per token, all SMs busy
  const int sms = num_sms(), g_min = sel_wide_min_g(p->cfg.max_ctx);
  if (!wide_ok || p->select_mode != HS_SELECT_AUTO || n < 1 || n > p->d.sel_ws_tokens || n * g_min > sms) return 0;
  int G = sms / n;
  if (G > SW_MAX_G) G = SW_MAX_G;
  const int g_want = (p->cfg.max_ctx + SW_TARGET - 1) / SW_TARGET;
  if (G > g_want) G = g_want > g_min ? g_want : g_min;
  return G;
}

uint32_t* select_hist0(hs_pool* p, int n, bool wide_ok) {
  if (n != 1 || select_wide_groups(p, n, wide_ok) == 0) return nullptr;
  return reinterpret_cast<SelWs*>(p->d.sel_ws)->hist[0];
}

hs_status launch_select(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                        int32_t* d_topk, cudaStream_t st, bool fp_keys, bool wide_ok, bool hist0_done) {
  const int G = select_wide_groups(p, n, wide_ok);
  if (G > 0) return launch_select_wide(p, n, scores, ld, d_limit, d_topk, fp_keys, G, hist0_done, st);
  // Many query tokens, at most one per SM: every token's keys in chunks over the whole
  // GPU (three launches, no cross-CTA waits), so the longest token no longer sets the
  // time of the launch. More tokens than SMs: one CTA per token, which then keeps every
  // SM busy. (Chunked measured faster at 128 tokens of 8K-241K keys, slower at 256
  // tokens of ~80K keys.)
  if (wide_ok && n > num_sms() / 8) {
    if (n <= p->d.bsel_tokens && n <= num_sms())
      return launch_select_batch(p, n, scores, ld, d_limit, d_topk, fp_keys, st);
    return launch_select_token(p, n, scores, ld, d_limit, d_topk, fp_keys, st);
  }
  // otherwise 16 CTAs per token: each CTA's chunk is smaller and every pass shorter
  return launch_select_cl<16>(p, n, scores, ld, d_limit, d_topk, fp_keys, st);
}

}  // namespace hs
