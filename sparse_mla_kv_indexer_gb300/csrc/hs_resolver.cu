// Fused top-K resolver and the single-row host -> pool copies of its misses.
//
// "vLLM introduces Hybrid HiSparse hybrid sparse offloading for GLM 5.3" (vLLM
// blog Part 1), section "How it works", hybrid residency: a fused kernel
// resolves the top-K; resident tokens are read in place, hot tokens are read and
// have their LRU entry refreshed, a miss copies a single row from pinned host
// memory into an LRU slot; the resolver hands the attention HMA row ids for
// resident and hot rows alike, and nothing on the decode path waits for a CPU
// decision. With MTP the verification tokens of a request resolve together.
//
// One CTA per request segment (the tokens of one request in the batch):
//   1. U = ascending union of the segment's selected tokens: each token's top-K is
//      ascending, so the rows are merged by rank (binary searches, one pass) and
//      repeats dropped; a single row is taken as it is;
//   2. classify each t in U: block table >= 0 -> RESIDENT; hot slot -> HIT
//      (stamp = step); else MISS;
//   3. victims = leased slots not hit this step, ordered by (stamp, slot): a
//      histogram over stamp values finds the threshold stamp, the victims are
//      compacted in slot order and bitonic-sorted by (stamp, slot);
//   4. misses (ascending token order) take victims in order; maps updated; each
//      consumed victim entry becomes that miss's copy record;
//   5. row ids and plan entries written for every (token, k);
//   6. the request's cluster of 8 CTAs copies each missed row of every layer of
//      the group from the mapped host pool into the slot's pool row, 16 bytes per
//      thread, reading the records from the resolving CTA's shared memory.
// Block tables, hot pages and the request ids are read before the wait on the
// preceding kernel (they do not depend on it); the block-table and token->slot
// entries of a thread's tokens are fetched in one round trip.
#include <climits>

#include "hs_internal.cuh"

namespace hs {

constexpr int RS_THREADS = 1024;
constexpr int RS_MAXU = 8192;        // max_q * topk <= 4 * 2048
constexpr int RS_HBINS = 1024;

enum Kind : int8_t { K_PAD = 0, K_RES = 1, K_HIT = 2, K_MISS = 3 };

__device__ __forceinline__ int rs_block_scan(int v, int* wt, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wt[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = wt[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    wt[lane] = t;
    if (lane == 31 && total) *total = t;
  }
  __syncthreads();
  int r = x - v + (warp ? wt[warp - 1] : 0);
  __syncthreads();
  return r;
}

// ascending bitonic sort of n (power of two) keys in shared memory
template <typename T>
__device__ void bitonic_sort(T* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int p = i ^ j;
        if (p > i) {
          T x = a[i], y = a[p];
          bool up = (i & k) == 0;
          if ((x > y) == up) { a[i] = y; a[p] = x; }
        }
      }
      __syncthreads();
    }
  }
}

constexpr int RS_COPY_CTAS = 8;      // CTAs of a request's cluster that copy its missed rows
constexpr int RS_COPY_UNROLL = 4;    // 16-byte host loads in flight per thread

// CL: CTAs per request segment (a thread-block cluster when CL > 1) that copy its
// missed rows; the first resolves.
template <int CL>
__global__ void __launch_bounds__(RS_THREADS, 1)
resolve_kernel(Dev D, int group, int step, int n_tok, const int32_t* __restrict__ req_of,
               const int32_t* __restrict__ topk, int32_t* __restrict__ row_ids, hs_plan_entry* __restrict__ plan) {
  extern __shared__ __align__(16) uint8_t rs_smem[];
  int32_t* U = reinterpret_cast<int32_t*>(rs_smem);                 // [RS_MAXU] union (then sorted)
  int32_t* info = U + RS_MAXU;                                      // [RS_MAXU] row (resident) or slot
  int32_t* evic = info + RS_MAXU;                                   // [RS_MAXU] evicted token
  int8_t* kind = reinterpret_cast<int8_t*>(evic + RS_MAXU);         // [RS_MAXU]
  // [RS_MAXU] victims (stamp + 1, slot); each, once taken by a miss, becomes that
  // miss's copy record (pool row, token)
  unsigned long long* V = reinterpret_cast<unsigned long long*>(kind + RS_MAXU);
  __shared__ int wt[32];
  __shared__ int s_tot, s_cnt[3], s_bin, s_before, s_min, s_listed, s_len[4];
  __shared__ uint32_t hbin[RS_HBINS];
  __shared__ int32_t s_hotp[256];                                   // hot pages of (request, group)

  const int b = blockIdx.x;
  const int rank = (int)blockIdx.y;          // rank in the request's cluster; 0 resolves, all copy
  const int K = D.topk;
  const int tid = threadIdx.x;
  const int lo_layer = group * D.lpi;
  const int n_lg = min(D.lpi, D.n_layers - lo_layer);

  // ---- prologue: everything that does not depend on the top-K being resolved.
  //      The request ids, block tables and hot state were written by the host or by
  //      earlier steps, before the preceding kernel started. ----
  const int r = req_of[b];
  int T = 1;
  bool first = true;
  {
    // up to 4 query tokens per request, plus one more to detect a longer run
    int nx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) nx[k] = b + 1 + k < n_tok ? req_of[b + 1 + k] : -2;
    if (b > 0 && req_of[b - 1] == r) first = false;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (T == k + 1 && nx[k] == r) T = k + 2;
  }
  const bool bad = r < 0 || r >= D.max_requests || T > D.max_q;
  if (!first) {            // not the first token of its request: the first one resolves the segment
    griddep_wait();
    griddep_launch();
    return;                // uniform across the cluster
  }
  const size_t rg = bad ? 0 : (size_t)r * D.n_groups + group;
  const int n_slots = bad ? 0 : min(D.n_hot[rg], D.hot_pages_max) * PAGE;
  if (rank == 0 && !bad)
    for (int k = tid; k < D.hot_pages_max; k += RS_THREADS) s_hotp[k] = D.hot_pages[rg * D.hot_pages_max + k];
  griddep_wait();
  griddep_launch();

  if (rank == 0) {
    if (tid == 0) s_listed = 0;
    if (bad) {
      if (tid == 0) set_status(D.status, HS_ERR_BAD_ID);
    } else {
      int32_t* stamp = D.slot_stamp + rg * D.hot_rows;
      int32_t* stok = D.slot_token + rg * D.hot_rows;
      int32_t* t2s = D.tok2slot + rg * D.max_ctx;
      const int32_t* btr = D.bt + (size_t)r * D.max_pages;

      // ---- 1. union of the selections ----
      const int n_in = T * K;
      int nU;
      if (T == 1) {
        for (int i = tid; i < K; i += RS_THREADS) {
          int t = topk[(size_t)b * K + i];
          if (t >= D.max_ctx) { set_status(D.status, HS_ERR_BAD_ID); t = -1; }
          U[i] = t;
        }
        __syncthreads();
        int c = 0;
        for (int i = tid; i < K; i += RS_THREADS) c += U[i] >= 0;
        c = __reduce_add_sync(0xffffffffu, c);
        if (tid == 0) s_tot = 0;
        __syncthreads();
        if ((tid & 31) == 0) atomicAdd(&s_tot, c);
        __syncthreads();
        nU = s_tot;     // pads are at the end of an ascending top-K row
      } else {
        // T rows of K entries, pads (and ids beyond the context) as INT_MAX
        int np = 1;
        while (np < n_in) np <<= 1;
        if (tid < 4) s_len[tid] = 0;
        for (int i = tid; i < np; i += RS_THREADS) {
          int t = i < n_in ? topk[(size_t)b * K + i] : -1;
          if (t >= D.max_ctx) { set_status(D.status, HS_ERR_BAD_ID); t = -1; }
          U[i] = t < 0 ? INT_MAX : t;
          info[i] = INT_MAX;
        }
        __syncthreads();
        // A top-K row is ascending with its pads at the end; each row's length is the
        // index of its first pad. Rows of that form are merged by rank; any other
        // input is sorted whole.
        int bad_row = 0;
        for (int i = tid; i < n_in; i += RS_THREADS) {
          const int k = i % K;
          const bool last = k == K - 1 || U[i + 1] == INT_MAX;
          if (k != K - 1 && U[i + 1] != INT_MAX && U[i] >= U[i + 1]) bad_row = 1;
          if (U[i] != INT_MAX && last) s_len[i / K] = k + 1;
        }
        const bool by_rank = !__syncthreads_or(bad_row);
        if (by_rank) {
          // An entry's place in the merged order is its index in its own row plus the
          // entries of the other rows before it: those < t, and those == t of earlier
          // rows (equal tokens keep row order, so every place is taken once).
          for (int i = tid; i < n_in; i += RS_THREADS) {
            const int j = i / K, k = i - j * K;
            if (k >= s_len[j]) continue;
            const int t = U[i];
            int pos = k;
            for (int o = 0; o < T; ++o) {
              if (o == j) continue;
              const int32_t* row = U + o * K;
              int lo = 0, hi = s_len[o];   // first entry > t (earlier rows) or >= t (later rows)
              while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (o < j ? row[mid] <= t : row[mid] < t) lo = mid + 1; else hi = mid;
              }
              pos += lo;
            }
            info[pos] = t;
          }
        } else {
          bitonic_sort(U, np);
        }
        __syncthreads();
        // drop repeats of the ascending sequence, keep the order
        const int32_t* srt = by_rank ? info : U;
        int32_t* dst = by_rank ? U : info;
        constexpr int IPT = RS_MAXU / RS_THREADS;
        int f[IPT], cnt = 0;
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
          int i = tid * IPT + k;
          f[k] = (i < np && srt[i] != INT_MAX && (i == 0 || srt[i] != srt[i - 1])) ? 1 : 0;
          cnt += f[k];
        }
        int pos = rs_block_scan(cnt, wt, &s_tot);
#pragma unroll
        for (int k = 0; k < IPT; ++k)
          if (f[k]) dst[pos++] = srt[tid * IPT + k];
        __syncthreads();
        nU = s_tot;
        if (!by_rank) {
          for (int i = tid; i < nU; i += RS_THREADS) U[i] = info[i];
          __syncthreads();
        }
      }

      // ---- 2. classify: block-table and token->slot entries of all of a thread's
      //         tokens are loaded together (one round trip) ----
      if (tid < 3) s_cnt[tid] = 0;
      __syncthreads();
      int n_res = 0, n_hit = 0, n_miss_l = 0;
      constexpr int CB = 2;   // tokens per thread per round trip (a single token's top-K takes one)
      for (int k0 = 0; k0 * RS_THREADS < nU; k0 += CB) {
        int pgv[CB], slv[CB];
#pragma unroll
        for (int k = 0; k < CB; ++k) {
          const int i = tid + (k0 + k) * RS_THREADS;
          const int t = i < nU ? U[i] : -1;
          pgv[k] = t >= 0 ? btr[t >> 6] : -1;
          slv[k] = t >= 0 ? t2s[t] : -1;
        }
#pragma unroll
        for (int k = 0; k < CB; ++k) {
          const int i = tid + (k0 + k) * RS_THREADS;
          if (i >= nU) break;
          const int t = U[i];
          evic[i] = -1;
          if (t < 0) { kind[i] = K_PAD; info[i] = -1; continue; }
          const int pg = pgv[k];
          if (pg >= 0) {
            if (pg >= D.num_pages) { set_status(D.status, HS_ERR_BAD_ID); kind[i] = K_PAD; info[i] = -1; continue; }
            kind[i] = K_RES;
            info[i] = pg * PAGE + (t & 63);
            ++n_res;
          } else {
            const int sl = slv[k];
            if (sl >= n_slots) { set_status(D.status, HS_ERR_BAD_ID); kind[i] = K_PAD; info[i] = -1; continue; }
            if (sl >= 0) {
              kind[i] = K_HIT;
              info[i] = sl;
              stamp[sl] = step;
              ++n_hit;
            } else {
              kind[i] = K_MISS;
              info[i] = -1;
              ++n_miss_l;
            }
          }
        }
      }
      n_res = __reduce_add_sync(0xffffffffu, n_res);
      n_hit = __reduce_add_sync(0xffffffffu, n_hit);
      n_miss_l = __reduce_add_sync(0xffffffffu, n_miss_l);
      if ((tid & 31) == 0) {
        atomicAdd(&s_cnt[0], n_res);
        atomicAdd(&s_cnt[1], n_hit);
        atomicAdd(&s_cnt[2], n_miss_l);
      }
      __threadfence_block();
      __syncthreads();
      const int n_miss = s_cnt[2];

      // ---- 3. victims ----
      if (n_miss > 0) {
        // candidates: leased slots whose stamp is not this step; smallest stamp first
        if (tid == 0) s_min = INT_MAX;
        __syncthreads();
        int lmin = INT_MAX, lcand = 0;
        for (int sl = tid; sl < n_slots; sl += RS_THREADS) {
          int st = stamp[sl];
          if (st != step) { lmin = min(lmin, st); ++lcand; }
        }
        lmin = __reduce_min_sync(0xffffffffu, lmin);
        lcand = __reduce_add_sync(0xffffffffu, lcand);
        if (tid == 0) s_tot = 0;
        __syncthreads();
        if ((tid & 31) == 0) { atomicMin(&s_min, lmin); atomicAdd(&s_tot, lcand); }
        __syncthreads();
        const int n_cand = s_tot;
        if (n_cand < n_miss) {
          if (tid == 0) set_status(D.status, HS_ERR_CAPACITY);
          for (int i = tid; i < nU; i += RS_THREADS)
            if (kind[i] == K_MISS) { kind[i] = K_PAD; }
        } else {
          // threshold stamp by histogram over stamp windows of RS_HBINS values
          long long wbase = s_min;
          int need = n_miss;
          int thr_stamp = 0, take_eq = 0;
          for (;;) {
            for (int i = tid; i < RS_HBINS; i += RS_THREADS) hbin[i] = 0;
            __syncthreads();
            for (int sl = tid; sl < n_slots; sl += RS_THREADS) {
              int st = stamp[sl];
              if (st != step && st >= wbase)
                atomicAdd(&hbin[(int)min((long long)st - wbase, (long long)RS_HBINS - 1)], 1u);
            }
            __syncthreads();
            int v = (int)hbin[tid];     // RS_HBINS == RS_THREADS
            int before = rs_block_scan(v, wt, nullptr);
            if (before < need && need <= before + v) { s_bin = tid; s_before = before; }
            __syncthreads();
            const int B = s_bin;
            if (B < RS_HBINS - 1) {
              thr_stamp = (int)(wbase + B);
              take_eq = need - s_before;
              break;
            }
            // the last bin lumps stamps >= wbase + RS_HBINS - 1: slide the window
            need -= s_before;
            wbase += RS_HBINS - 1;
            if (wbase > step) {   // cannot happen: stamps never exceed step
              thr_stamp = step;
              take_eq = need;
              break;
            }
            __syncthreads();
          }
          // flag victims in slot order: stamp < thr, or == thr among the first take_eq
          constexpr int SPT = 16;     // slots per thread (hot_rows <= 16384)
          int lo_s = tid * SPT;
          int eqc = 0;
          for (int k = 0; k < SPT; ++k) {
            int sl = lo_s + k;
            if (sl < n_slots && stamp[sl] == thr_stamp) ++eqc;
          }
          int eq_before = rs_block_scan(eqc, wt, nullptr);
          int vf = 0, vc = 0;
          for (int k = 0; k < SPT; ++k) {
            int sl = lo_s + k;
            if (sl >= n_slots) break;
            int st = stamp[sl];
            bool vic = false;
            if (st != step) {
              if (st < thr_stamp) vic = true;
              else if (st == thr_stamp) { vic = eq_before < take_eq; ++eq_before; }
            }
            vf |= (vic ? 1 : 0) << k;
            vc += vic;
          }
          int vpos = rs_block_scan(vc, wt, nullptr);
          for (int k = 0; k < SPT; ++k)
            if (vf >> k & 1) {
              int sl = lo_s + k;
              if (vpos < RS_MAXU) V[vpos] = ((unsigned long long)(uint32_t)(stamp[sl] + 1) << 32) | (uint32_t)sl;
              ++vpos;
            }
          int np = 1;
          while (np < n_miss) np <<= 1;
          for (int i = n_miss + tid; i < np; i += RS_THREADS) V[i] = ~0ull;
          __syncthreads();
          bitonic_sort(V, np);
          // ---- 4. misses in ascending token order take victims in order ----
          constexpr int IPT = RS_MAXU / RS_THREADS;
          int mf = 0, mc = 0;
          for (int k = 0; k < IPT; ++k) {
            int i = tid * IPT + k;
            if (i < nU && kind[i] == K_MISS) { mf |= 1 << k; ++mc; }
          }
          int mpos = rs_block_scan(mc, wt, nullptr);
          const int64_t* hpr = D.host_pg + (size_t)r * D.max_pages;
          for (int k = 0; k < IPT; ++k) {
            if (!(mf >> k & 1)) continue;
            int i = tid * IPT + k;
            int t = U[i];
            int v = (int)(uint32_t)(V[mpos] & 0xffffffffu);
            unsigned long long rec = ~0ull;   // copy record: (pool row, token); none when invalid
            if (v < 0 || v >= n_slots) {      // cannot happen when exactly n_miss victims were flagged
              set_status(D.status, HS_ERR_CAPACITY);
              kind[i] = K_PAD;
            } else {
              int old = stok[v];
              if (old >= 0) t2s[old] = -1;
              stok[v] = t;
              stamp[v] = step;
              t2s[t] = v;
              info[i] = v;
              evic[i] = old;
              const int64_t hp = hpr[t >> 6];
              const int hpage = s_hotp[v >> 6];
              if (hp < 0 || hp >= D.host_pages) set_status(D.status, HS_ERR_HOST_MISSING);
              else if (hpage < 0 || hpage >= D.num_pages) set_status(D.status, HS_ERR_BAD_ID);
              else rec = ((unsigned long long)(uint32_t)(hpage * PAGE + (v & 63)) << 32) | (uint32_t)t;
            }
            V[mpos] = rec;   // this victim is consumed by this miss alone
            ++mpos;
          }
          if (tid == 0) s_listed = n_miss;
        }
      }
      __syncthreads();
      if (tid == 0) {
        atomicAdd(&D.counters[C_RESIDENT], (unsigned long long)s_cnt[0]);
        atomicAdd(&D.counters[C_HITS], (unsigned long long)s_cnt[1]);
        atomicAdd(&D.counters[C_MISSES], (unsigned long long)n_miss);
        atomicAdd(&D.counters[C_H2D], (unsigned long long)s_listed * n_lg * ROW);
      }

      // ---- 5. row ids and plan, from shared memory ----
      for (int e = tid; e < T * K; e += RS_THREADS) {
        const size_t o = (size_t)b * K + e;
        int t, i;
        if (T == 1) {
          i = e;
          t = e < nU ? U[e] : -1;
        } else {
          t = topk[o];
          int lo = 0, hi = nU - 1;
          while (lo < hi) {
            int mid = (lo + hi) >> 1;
            if (U[mid] < t) lo = mid + 1; else hi = mid;
          }
          i = lo;
        }
        int kd = K_PAD, slot = -1, row = -1, ev = -1;
        if (t >= 0 && t < D.max_ctx) {
          kd = i < nU ? kind[i] : K_PAD;
          if (kd == K_RES) {
            row = info[i];
          } else if (kd == K_HIT || kd == K_MISS) {
            slot = info[i];
            const int hpage = s_hotp[slot >> 6];
            row = (hpage >= 0 && hpage < D.num_pages) ? hpage * PAGE + (slot & 63) : -1;
            ev = evic[i];
          }
        }
        row_ids[o] = row;
        if (plan) {
          hs_plan_entry pe;
          pe.kind = kd;
          pe.slot = slot;
          pe.row = row;
          pe.evicted = ev;
          plan[o] = pe;
        }
      }
    }
  }

  // ---- 6. every CTA of the cluster copies its share of the missed rows of every
  //         layer of the group from the mapped host pool (records in rank 0) ----
  if constexpr (CL > 1) cluster_sync();   // rank 0's records are complete
  else __syncthreads();
  const int n_rec = CL > 1 ? (int)ld_cluster_u32(mapa(smem_u32(&s_listed), 0)) : s_listed;
  if (n_rec > 0) {
    const uint32_t recs = CL > 1 ? mapa(smem_u32(V), 0) : 0u;
    const int64_t* hpr = D.host_pg + (size_t)r * D.max_pages;
    const long long total = (long long)n_rec * n_lg * ROW_CHUNKS;
    const long long stride = (long long)CL * RS_THREADS;
    for (long long c0 = (long long)rank * RS_THREADS + tid; c0 < total; c0 += stride * RS_COPY_UNROLL) {
      uint4 v[RS_COPY_UNROLL];
      uint8_t* dst[RS_COPY_UNROLL];
#pragma unroll
      for (int u = 0; u < RS_COPY_UNROLL; ++u) {   // all host loads in flight, then the stores
        const long long c = c0 + u * stride;
        dst[u] = nullptr;
        if (c >= total) continue;
        const long long row_i = c / ROW_CHUNKS;
        const int part = (int)(c - row_i * ROW_CHUNKS);
        const int m = (int)(row_i / n_lg);
        const int layer = lo_layer + (int)(row_i - (long long)m * n_lg);
        const unsigned long long rec = CL > 1 ? ld_cluster_u64(recs + 8u * (uint32_t)m) : V[m];
        if (rec == ~0ull) continue;
        const int t = (int)(uint32_t)rec, prow = (int)(rec >> 32);
        const int64_t hp = hpr[t >> 6];
        v[u] = *reinterpret_cast<const uint4*>(D.host + ((size_t)(hp * D.n_layers + layer) * PAGE + (t & 63)) * ROW +
                                               part * 16);
        dst[u] = D.kv[layer] + (size_t)prow * ROW + part * 16;
      }
#pragma unroll
      for (int u = 0; u < RS_COPY_UNROLL; ++u)
        if (dst[u]) *reinterpret_cast<uint4*>(dst[u]) = v[u];
    }
  }
  if constexpr (CL > 1) cluster_sync();   // rank 0's shared memory is read by its peers until here
}

constexpr int RS_SMEM = RS_MAXU * (4 + 4 + 4 + 1 + 8);

hs_status launch_resolve(hs_pool* p, int group, int step, int n, const int32_t* d_req, const int32_t* d_topk,
                         int32_t* d_row_ids, hs_plan_entry* d_plan, cudaStream_t st) {
  // Few query tokens: one cluster of RS_COPY_CTAS CTAs per token (the first token of
  // each request resolves it, the cluster copies its misses). Many tokens: one CTA per
  // token, so that every request resolves in the same wave of CTAs (a CTA takes a
  // whole SM's shared memory).
  if ((long long)n * RS_COPY_CTAS <= num_sms()) {
    if (ensure_kernel_attrs(resolve_kernel<RS_COPY_CTAS>, RS_SMEM) != HS_OK) return HS_ERR_CUDA;
    return launch_pdl_cluster(resolve_kernel<RS_COPY_CTAS>, dim3(n, RS_COPY_CTAS), dim3(RS_THREADS), RS_SMEM, st,
                              dim3(1, RS_COPY_CTAS, 1), p->d, group, step, n, d_req, d_topk, d_row_ids, d_plan);
  }
  if (ensure_kernel_attrs(resolve_kernel<1>, RS_SMEM) != HS_OK) return HS_ERR_CUDA;
  return launch_pdl(resolve_kernel<1>, dim3(n, 1), dim3(RS_THREADS), RS_SMEM, st, 0, p->d, group, step, n, d_req,
                    d_topk, d_row_ids, d_plan);
}

// Replay: each (token, k) looked up in the residency maps as they stand; read only.
__global__ void __launch_bounds__(256)
replay_kernel(Dev D, int group, int n_tok, const int32_t* __restrict__ req_of, const int32_t* __restrict__ topk,
              int32_t* __restrict__ row_ids) {
  griddep_wait();
  griddep_launch();
  const int K = D.topk;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)n_tok * K) return;
  const int j = (int)(e / K);
  const int r = req_of[j];
  const int t = topk[e];
  int row = -1;
  if (r < 0 || r >= D.max_requests || t >= D.max_ctx) {
    set_status(D.status, HS_ERR_BAD_ID);
  } else if (t >= 0) {
    const size_t rg = (size_t)r * D.n_groups + group;
    const int pg = D.bt[(size_t)r * D.max_pages + (t >> 6)];
    if (pg >= 0 && pg < D.num_pages) {
      row = pg * PAGE + (t & 63);
    } else {
      const int n_slots = min(D.n_hot[rg], D.hot_pages_max) * PAGE;
      const int sl = D.tok2slot[rg * D.max_ctx + t];
      const int hpage = (sl >= 0 && sl < n_slots) ? D.hot_pages[rg * D.hot_pages_max + (sl >> 6)] : -1;
      if (hpage >= 0 && hpage < D.num_pages) row = hpage * PAGE + (sl & 63);
      else set_status(D.status, HS_ERR_NOT_RESOLVED);
    }
  }
  row_ids[e] = row;
}

hs_status launch_replay(hs_pool* p, int group, int n, const int32_t* d_req, const int32_t* d_topk, int32_t* d_row_ids,
                        cudaStream_t st) {
  const long long total = (long long)n * p->cfg.topk;
  return launch_pdl(replay_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, st, 0, p->d, group, n, d_req,
                    d_topk, d_row_ids);
}

}  // namespace hs
