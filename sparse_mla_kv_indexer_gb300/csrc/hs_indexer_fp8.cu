// FP8 indexer scoring for key caches in the pages' format.
//
// "Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse" (vLLM blog Part 2),
// footnote 3: an indexer key is 128 FP8 values plus a 4-byte scale (132 bytes).
// Score of earlier token t for a query token:
//   s[t] = scale_t * sum_h w[h] * max(0, sum_d q[h][d] * k_t[d])      (fp32)
// with q and k in e4m3 and the query's own scale folded into its head weights w.
//
// One persistent CTA per SM, ten warps:
//  * warp 8 (producer) fetches page ids 32 tiles ahead and loads each 128-key
//    tile with two 2-D tensor loads (TMA), one per 64-key page: the e4m3 key rows
//    land 128-byte swizzled, which is exactly the K-major operand layout of
//    tcgen05.mma, so there is no conversion stage; the pages' 64 fp32 scales
//    come with a 256-byte bulk copy each into a ring of their own, so that a key
//    stage is free as soon as its MMAs complete (the MMA commit releases it) and
//    only the small scale slot waits for the epilogue;
//  * warp 9 puts each request segment's queries (e4m3, swizzled) in place, once
//    its earlier MMAs have completed, and issues tcgen05.mma kind::f8f6f4 (M = 128
//    keys, N = T * H_i, K = 128 in four steps of 32) straight from the stage ring
//    into up to 8 TMEM accumulators;
//  * warps 0-7 (epilogue, two warpgroups taking alternate tiles, so one tile's
//    TMEM read and barrier latency overlaps the other's) read the accumulators,
//    form the fp32 score and store it as an order-preserving integer key for the
//    top-K selection (and as fp32 when the caller asks), then release the
//    accumulator and the stage.
#include "hs_select.cuh"

namespace hs {

constexpr int F8_THREADS = 320;
constexpr int F8_EPI_GROUPS = 2;                      // epilogue warpgroups
constexpr int F8_PRODUCER_WARP = 8, F8_MMA_WARP = 9;
constexpr int F8_TILE = 128;                          // keys per tile (two pages)
constexpr int F8_KEY_BYTES = F8_TILE * IDX_DIM;       // 16 KB of e4m3 keys
constexpr int F8_STAGE = F8_KEY_BYTES;                // a key stage; 1 KB aligned
constexpr int F8_MAX_STAGES = 12;
constexpr int F8_SC_SLOTS = 16;                       // scale ring: 128 fp32 per slot
constexpr int F8_SC_BYTES = F8_SC_SLOTS * F8_TILE * 4;
constexpr int F8_MAX_ACC = 8;
constexpr int F8_TMEM_COLS = 512;
constexpr int F8_BUDGET = 227 * 1024;
constexpr int F8_PAGE_ROWS = HS_IDX_FP8_PAGE_BYTES / 128;   // a page is 66 rows of 128 bytes
static_assert(F8_SC_SLOTS % 2 == 0, "each scale slot stays with one epilogue warpgroup");
constexpr int F8_N_BARS = 2 * F8_MAX_STAGES + 2 * F8_MAX_ACC + 2 * F8_SC_SLOTS + 1;
static_assert(F8_N_BARS * 8 + 32 <= 1024, "barriers and flags fit their region");

struct F8Layout {
  int b_bytes;     // query operand [N][128] e4m3 (128-byte swizzled), 1 KB aligned
  int off_stage, stages, off_sc, off_bar, off_seg, off_hist, smem;   // off_hist: 0 = no histogram
  int acc_cols, n_acc;
};

static F8Layout f8_layout(int n_max_rows, int max_tokens, bool hist) {
  F8Layout L;
  L.b_bytes = (n_max_rows * 128 + 1023) & ~1023;
  L.off_stage = L.b_bytes;
  const int hist_bytes = hist ? SEL_BINS * 4 : 0;
  const int tail = F8_SC_BYTES + 1024 + max_tokens * 16 + F8_EPI_GROUPS * 4 * 64 * 4 + 2 * max_tokens * 4 +
                   hist_bytes + 1024;
  const int st = (F8_BUDGET - L.off_stage - tail) / F8_STAGE;
  L.stages = st > F8_MAX_STAGES ? F8_MAX_STAGES : st;
  L.off_sc = L.off_stage + L.stages * F8_STAGE;
  L.off_bar = L.off_sc + F8_SC_BYTES;
  L.off_seg = L.off_bar + 1024;
  L.off_hist = hist ? L.off_seg + max_tokens * 16 + F8_EPI_GROUPS * 4 * 64 * 4 + 2 * max_tokens * 4 : 0;
  L.smem = L.off_seg + max_tokens * 16 + F8_EPI_GROUPS * 4 * 64 * 4 + 2 * max_tokens * 4 + hist_bytes + 1024;
  L.acc_cols = 32;
  while (L.acc_cols < n_max_rows) L.acc_cols <<= 1;
  L.n_acc = F8_TMEM_COLS / L.acc_cols < F8_MAX_ACC ? F8_TMEM_COLS / L.acc_cols : F8_MAX_ACC;
  return L;
}

struct F8Seg {
  int32_t first, ntok, maxlim, tile_end;
};

// Order-preserving integer of an fp32 (finite): the top-K selection works on it.
__device__ __forceinline__ long long f32_order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (long long)((u & 0x80000000u) ? ~u : (u | 0x80000000u));
}

__device__ __forceinline__ void f8_named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier over n threads that also ORs a flag across them: every thread
// leaves with the same answer, so an error seen by one thread ends the loop of all.
__device__ __forceinline__ int f8_sync_or(int id, int n, int flag) {
  int out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}"
      : "=r"(out) : "r"(flag), "r"(id), "r"(n) : "memory");
  return out;
}
__device__ __forceinline__ void f8_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(F8_THREADS, 1)
indexer_fp8_kernel(Dev D, const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap2,
                   const __grid_constant__ CUtensorMap smap2, int il, int n_tok,
                   const int32_t* __restrict__ req_of, const int32_t* __restrict__ limit_of,
                   const uint8_t* __restrict__ qg, const float* __restrict__ wg, long long* __restrict__ keys_out,
                   float* __restrict__ scores_out, int ld, F8Layout L, uint32_t* __restrict__ hist0) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NS = L.stages;
  uint8_t* Bq = smem;                                            // queries
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* full = bars;                                         // [NS] stage loaded
  uint64_t* empty = bars + F8_MAX_STAGES;                        // [NS] stage's MMAs completed
  uint64_t* t_full = bars + 2 * F8_MAX_STAGES;                   // [n_acc]
  uint64_t* t_empty = t_full + F8_MAX_ACC;                       // [n_acc]
  uint64_t* c_full = t_empty + F8_MAX_ACC;                       // [F8_SC_SLOTS] scales loaded
  uint64_t* c_empty = c_full + F8_SC_SLOTS;                      // [F8_SC_SLOTS] scales read by the epilogue
  uint64_t* b_done = c_empty + F8_SC_SLOTS;                      // [1] MMAs reading the queries completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_done + 1);
  int32_t* s_nseg = reinterpret_cast<int32_t*>(tmem_slot + 1);
  int32_t* s_dead = s_nseg + 1;
  int32_t* s_issued = s_nseg + 2;
  F8Seg* segs = reinterpret_cast<F8Seg*>(smem + L.off_seg);
  float* s_w = reinterpret_cast<float*>(segs + D.max_tokens);     // [F8_EPI_GROUPS][4][64]
  int32_t* s_req = reinterpret_cast<int32_t*>(s_w + F8_EPI_GROUPS * 4 * 64);   // [n_tok]
  int32_t* s_lim = s_req + D.max_tokens;                          // [n_tok]
  // hist0 (one query token, wide selection): the selection's level-0 histogram of
  // this CTA's keys, added to the selection's global sums at the end
  uint32_t* s_hist = hist0 ? reinterpret_cast<uint32_t*>(smem + L.off_hist) : nullptr;   // [SEL_BINS]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hi = D.n_idx_heads;
  const int8_t* keys = D.idx[il];

  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), F8_TMEM_COLS);
  if (tid == 0) {
    for (int b = 0; b < F8_N_BARS; ++b) mbar_init(smem_u32(&bars[b]), 1);
    fence_mbar_init();
  }
  if (s_hist)
    for (int b = tid; b < SEL_BINS; b += F8_THREADS) s_hist[b] = 0;
  // Request ids, limits, queries, weights and the index block table are inputs,
  // final before the preceding kernel started: the segments, page ids, query operand
  // and weights are set up while it finishes. The producer waits for that kernel
  // before its first key copy (the keys may have been appended by it); the score and
  // histogram writes follow the copies.
  // ---- request segments of the batch (tokens of one request are contiguous) ----
  for (int t = tid; t < n_tok; t += F8_THREADS) {
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
      F8Seg& sg = segs[ns - 1];
      sg.ntok++;
      sg.maxlim = max(sg.maxlim, s_lim[t]);
    }
    for (int i = 0; i < ns; ++i) {
      tiles += (segs[i].maxlim + F8_TILE - 1) / F8_TILE;
      segs[i].tile_end = tiles;
    }
    *s_nseg = ns;
    *s_dead = 0;
    *s_issued = 0;
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
      const int mid = (lo + hi) >> 1;
      if (segs[mid].tile_end > item) hi = mid; else lo = mid + 1;
    }
    return lo;
  };
  auto item_of = [&](int i) { return runs ? first_item + i : first_item + i * (int)gridDim.x; };

  if (warp == F8_PRODUCER_WARP) {
    // ------------------------------ producer ------------------------------
    // lane l holds the page ids of tile (32c + l) of the current and the next chunk
    auto fetch = [&](int i, int& p0, int& p1) {
      p0 = p1 = -2;
      if (i < n_local) {
        const int item = item_of(i);
        const int sg = seg_of(item);
        const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
        const int32_t* bt = D.idx_bt + (size_t)s_req[segs[sg].first] * D.max_pages + tile * 2;
        p0 = bt[0];
        p1 = ((tile * F8_TILE + PAGE) < segs[sg].maxlim) ? bt[1] : -2;   // -2: page beyond the limit
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
        const int rs = i % NS, cs = i % F8_SC_SLOTS;
        if (i >= NS && !mbar_wait_spin(smem_u32(&empty[rs]), ((i / NS) - 1) & 1, D.status)) *s_dead = 1;
        if (i >= F8_SC_SLOTS && !mbar_wait_spin(smem_u32(&c_empty[cs]), ((i / F8_SC_SLOTS) - 1) & 1, D.status))
          *s_dead = 1;
        dead = *(volatile int32_t*)s_dead;
        if (!dead) {
          const uint32_t bar = smem_u32(&full[rs]), cbar = smem_u32(&c_full[cs]);
          uint8_t* stage = smem + L.off_stage + rs * F8_STAGE;
          uint8_t* slot = smem + L.off_sc + cs * F8_TILE * 4;
          const int ips[2] = {ip0, ip1};
          uint32_t bytes = 0;
          for (int k = 0; k < 2; ++k) {
            if (ips[k] == -2) continue;
            if (ips[k] < 0 || ips[k] >= D.num_idx_pages) { set_status(D.status, HS_ERR_BAD_ID); continue; }
            bytes += PAGE * IDX_DIM;
          }
          mbar_expect_tx(bar, bytes);
          mbar_expect_tx(cbar, bytes / IDX_DIM * 4);
          // Copies take about the same time whatever their size up to 16-32 KB (the
          // SM's copy engine serialises them), so two adjacent pages -- the usual case,
          // a request's always-resident key cache is allocated in runs -- come with one
          // 3-D tensor load for their key rows and one 2-D load for their scales.
          const bool ok0 = ips[0] >= 0 && ips[0] < D.num_idx_pages, ok1 = ips[1] >= 0 && ips[1] < D.num_idx_pages;
          if (ok0 && ok1 && ips[1] == ips[0] + 1) {
            tma_load_3d(smem_u32(stage), &tmap2, 0, 0, ips[0], bar);
            tma_load_2d(smem_u32(slot), &smap2, 0, ips[0], cbar);
          } else {
            for (int k = 0; k < 2; ++k)
              if (k == 0 ? ok0 : ok1) {
                tma_load_2d(smem_u32(stage + k * PAGE * IDX_DIM), &tmap, 0, ips[k] * F8_PAGE_ROWS, bar);
                bulk_g2s(smem_u32(slot + k * PAGE * 4),
                         keys + (size_t)ips[k] * HS_IDX_FP8_PAGE_BYTES + PAGE * IDX_DIM, PAGE * 4, cbar);
              }
          }
          *s_issued = i + 1;
        }
      }
      if (__shfl_sync(0xffffffffu, dead, 0)) break;
    }
  } else if (warp == F8_MMA_WARP) {
    // ------------------------------ MMA issuer ------------------------------
    // lane 0 waits and issues; the warp's 32 lanes load each segment's queries
    int cur_seg = -1, nb = 0, any = 0;
    for (int i = 0; i < n_local; ++i) {
      const int rs = i % NS, tb = i % L.n_acc;
      const int sg = seg_of(item_of(i));
      int ok = 1;
      if (sg != cur_seg) {
        if (i > 0) {   // the previous segment's MMAs still read the query operand
          if (lane == 0) {
            umma_commit(smem_u32(b_done));
            ok = mbar_wait_spin(smem_u32(b_done), nb & 1, D.status);
          }
          ++nb;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) { *s_dead = 1; break; }
        }
        const F8Seg S = segs[sg];
        const int N = ((S.ntok * Hi) + 15) & ~15;
        for (int c = lane; c < N * 8; c += 32) {
          const int r = c >> 3, ch = c & 7;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < S.ntok * Hi) {
            const int j = r / Hi, h = r - j * Hi;
            v = *reinterpret_cast<const uint4*>(qg + ((size_t)(S.first + j) * Hi + h) * IDX_DIM + ch * 16);
          }
          *reinterpret_cast<uint4*>(Bq + sw128_chunk(r, ch)) = v;
        }
        fence_proxy_async();
        __syncwarp();
        cur_seg = sg;
      }
      if (lane == 0) {
        ok = mbar_wait_spin(smem_u32(&full[rs]), (i / NS) & 1, D.status);
        if (ok && i >= L.n_acc) ok = mbar_wait_spin(smem_u32(&t_empty[tb]), ((i / L.n_acc) - 1) & 1, D.status);
        if (ok && !*(volatile int32_t*)s_dead) {
          tc_fence_after();
          const int N = ((segs[sg].ntok * Hi) + 15) & ~15;
          const uint32_t idesc = idesc_f8_e4m3(128, N);
          const uint32_t a0 = smem_u32(smem + L.off_stage + rs * F8_STAGE), b0 = smem_u32(Bq);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {   // K = 128 e4m3 = one 128-byte swizzle atom, 32 per step
            const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b0 + kk * 32, 16, 1024);
            umma_f8(tmem + tb * L.acc_cols, ad, bd, idesc, kk > 0);
          }
          umma_commit(smem_u32(&t_full[tb]));
          umma_commit(smem_u32(&empty[rs]));        // the key stage is free once these MMAs complete
          any = 1;
        } else {
          ok = 0;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) { *s_dead = 1; break; }
    }
    if (lane == 0 && any && *(volatile int32_t*)s_dead) {
      // the epilogue may have stopped early: let the MMAs in flight finish before TMEM is freed
      umma_commit(smem_u32(b_done));
      mbar_wait_spin(smem_u32(b_done), nb & 1, D.status);
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int grp = warp >> 2, et = tid & 127;          // warpgroup, thread within it
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float* sw = s_w + grp * 4 * 64;
    int cur_seg = -1;
    for (int i = grp; i < n_local; i += F8_EPI_GROUPS) {
      const int item = item_of(i);
      const int sg = seg_of(item);
      const F8Seg S = segs[sg];
      const int tile = item - (sg ? segs[sg - 1].tile_end : 0);
      const int row = et;                        // TMEM lane = key row of the tile
      const int key = tile * F8_TILE + row;
      const int cs = i % F8_SC_SLOTS, tb = i % L.n_acc;
      if (sg != cur_seg) {
        f8_named_sync(2 + grp, 128);
        for (int c = et; c < 4 * 64; c += 128) {
          const int j = c >> 6, h = c & 63;
          sw[c] = (j < S.ntok && h < Hi) ? wg[(size_t)(S.first + j) * Hi + h] : 0.f;
        }
        f8_named_sync(2 + grp, 128);
        cur_seg = sg;
      }
      // a failed wait is recorded and the tile run through without stores, so that the
      // warpgroup's decision to stop is taken together at the barrier below
      int ok = mbar_wait_spin(smem_u32(&t_full[tb]), (i / L.n_acc) & 1, D.status);
      // a scale slot is refilled only after this warpgroup releases it, so its phase is this tile's
      ok = ok && mbar_wait_spin(smem_u32(&c_full[cs]), (i / F8_SC_SLOTS) & 1, D.status);
      if (!ok) *s_dead = 1;
      tc_fence_after();
      const float scale = *reinterpret_cast<const float*>(smem + L.off_sc + cs * F8_TILE * 4 + row * 4);
      for (int j = 0; j < S.ntok; ++j) {
        const int lim = s_lim[S.first + j];
        const uint32_t col0 = lane_base + (uint32_t)(tb * L.acc_cols + j * Hi);
        uint32_t r[64];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q * 16 < Hi) tmem_ld16(col0 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(r + q * 16));
        tmem_wait_ld();
        float a4[4] = {0.f, 0.f, 0.f, 0.f};      // four independent chains
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q * 16 < Hi) {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const float4 w4 = *reinterpret_cast<const float4*>(sw + j * 64 + q * 16 + k4 * 4);
              const float w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) a4[k] = fmaf(w[k], fmaxf(__uint_as_float(r[q * 16 + k4 * 4 + k]), 0.f), a4[k]);
            }
          }
        const float s = ((a4[0] + a4[1]) + (a4[2] + a4[3])) * scale + 0.f;   // + 0: a zero score is +0
        if (ok && key < lim) {
          const long long ok32 = f32_order_key(s);
          keys_out[(size_t)(S.first + j) * ld + key] = ok32;
          if (scores_out) scores_out[(size_t)(S.first + j) * ld + key] = s;
          if (s_hist) atomicAdd(&s_hist[bucket_of(sel_key(ok32, key), true)], 1u);
        }
      }
      tc_fence_before();
      const int dead = f8_sync_or(2 + grp, 128, *(volatile int32_t*)s_dead);
      if (dead) break;
      if (et == 0) {
        f8_arrive(smem_u32(&t_empty[tb]));
        f8_arrive(smem_u32(&c_empty[cs]));
      }
    }
    if (s_hist) {   // both warpgroups are done: this CTA's histogram to the global sums
      f8_named_sync(4, F8_EPI_GROUPS * 128);
      for (int b = tid; b < SEL_BINS; b += F8_EPI_GROUPS * 128)
        if (s_hist[b]) atomicAdd(&hist0[b], s_hist[b]);
    }
  }
  __syncthreads();
  if (*s_dead && tid == F8_PRODUCER_WARP * 32) {
    // drain the copies that may still be in flight (the last use of every stage
    // and scale slot) before the CTA's shared memory goes away
    for (int k = max(0, *s_issued - NS); k < *s_issued; ++k) mbar_wait_spin(smem_u32(&full[k % NS]), (k / NS) & 1, D.status);
    for (int k = max(0, *s_issued - F8_SC_SLOTS); k < *s_issued; ++k)
      mbar_wait_spin(smem_u32(&c_full[k % F8_SC_SLOTS]), (k / F8_SC_SLOTS) & 1, D.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, F8_TMEM_COLS);
}

hs_status launch_indexer_fp8(hs_pool* p, int il, int n, const int32_t* d_req, const int32_t* d_limit,
                             const uint8_t* d_q, const float* d_w, int64_t* d_keys, float* d_scores,
                             uint32_t* d_hist0, cudaStream_t st) {
  const int n_max = ((p->cfg.max_q_per_req * p->cfg.n_idx_heads) + 15) & ~15;
  const F8Layout L = f8_layout(n_max, p->cfg.max_tokens, d_hist0 != nullptr);
  // alternate tiles go to alternate epilogue warpgroups: an even accumulator count
  // keeps every accumulator with one warpgroup, so its phase waits never alias
  if (L.stages < 2 || L.n_acc % F8_EPI_GROUPS || il < 0 || 3 * il + 2 >= (int)p->idx_tmaps.size()) return HS_ERR_INVALID;
  if (ensure_kernel_attrs(indexer_fp8_kernel, L.smem) != HS_OK) return HS_ERR_CUDA;
  return launch_pdl(indexer_fp8_kernel, dim3(num_sms()), dim3(F8_THREADS), L.smem, st, 0, p->d,
                    p->idx_tmaps[3 * il], p->idx_tmaps[3 * il + 1], p->idx_tmaps[3 * il + 2], il, n, d_req, d_limit, d_q, d_w, reinterpret_cast<long long*>(d_keys), d_scores,
                    p->cfg.max_ctx, L, d_hist0);
}

}  // namespace hs
