// Top-K selection spread over the whole GPU, for batches of few query tokens.
//
// "vLLM introduces Hybrid HiSparse hybrid sparse offloading for GLM 5.3" (vLLM
// blog Part 1), section "Sparsity when you need it": each query token keeps the
// top-K (2,048) of the indexer scores of all earlier tokens. Ties go to the lower
// token index and the output is in ascending token order (keys in hs_select.cuh).
//
// One group of G CTAs per query token, all resident at once: at most one CTA per
// SM (the shared memory of a CTA rules out a second one) and n_tokens x G <= SMs.
// CTA g holds a contiguous chunk of the token's keys in shared memory.
//  * Levels of 4,096-bin histograms narrow the key range that holds the K-th
//    largest key. Each CTA adds its histogram to the token's sums in global
//    memory; a grid barrier (an arrival counter in global memory, every wait
//    bounded) publishes them; every CTA reads the same sums and takes the same
//    decision. Level 0 uses the buckets of the cluster selection, each further
//    level splits the range into 4,096 parts, until at most 4,096 keys are left.
//  * The CTAs append the keys of that range to a global list and publish how many
//    of their own keys lie above it. After one more barrier every CTA finds tau
//    (the K-th largest key) in the list by itself, adds the counts of the CTAs
//    before it to get its output offset, and writes its selected tokens in order.
//  * After the last barrier each CTA clears a share of the sums for the next launch.
//  * With a single query token the scoring kernel adds its CTAs' level-0 histograms
//    to the sums as it writes the scores (hist0_done), so the selection starts from
//    complete sums: no histogram pass over its chunk and no first barrier.
// Its successor may start launching only once every CTA is resident (after the
// first barrier), so a dependent kernel cannot take the SM a CTA still waits for.
#include "hs_select.cuh"

namespace hs {

namespace {

// Grid barrier of the G CTAs of one query token: wait until the arrival counter
// reaches `target`. After WAIT_NS the status records HS_ERR_TIMEOUT and false is
// returned to every thread of the CTA.
__device__ bool sw_barrier(unsigned long long* ctr, unsigned long long target, int32_t* status, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
    int ok = 1;
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if ((it & 63u) == 0) {
        const uint64_t now = globaltimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > WAIT_NS) {
          set_status(status, HS_ERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Bin of 4,096 counts (shared memory, or global sums read through L2) that holds
// the need-th largest key, scanning from the top: sets *s_bin and *s_above (the
// keys in higher bins).
template <bool GLOBAL>
__device__ void sw_find(const uint32_t* h, int need, int* warp_tot, int* s_bin, long long* s_above) {
  constexpr int PER = SEL_BINS / SW_THREADS;
  static_assert(PER == 8, "two 16-byte loads per thread");
  const int tid = threadIdx.x;
  // thread tid holds bins 4095 - 8 tid down to 4088 - 8 tid: t[k] = bin 4095 - 8 tid - k
  const uint4* hv = reinterpret_cast<const uint4*>(h + SEL_BINS - PER * (tid + 1));
  const uint4 lo4 = GLOBAL ? __ldcg(hv) : hv[0], hi4 = GLOBAL ? __ldcg(hv + 1) : hv[1];
  const uint32_t t[PER] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};
  int local = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) local += (int)t[k];
  if (tid == 0) {
    *s_bin = 0;
    *s_above = 0;
  }
  const int before = block_excl_scan(local, warp_tot, nullptr);
  if (before < need && need <= before + local) {
    int cum = before;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      if (cum + (int)t[k] >= need) {
        *s_bin = SEL_BINS - 1 - (tid * PER + k);
        *s_above = cum;
        break;
      }
      cum += (int)t[k];
    }
  }
  __syncthreads();
}

__device__ __forceinline__ bool in_range(unsigned long long k, unsigned long long base, unsigned long long width) {
  return k >= base && k - base < width;
}

__global__ void __launch_bounds__(SW_THREADS, 1)
select_wide_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
                   int32_t* __restrict__ topk, int fp_keys, int G, int hist0_done) {
  const int tok = blockIdx.x / G, g = blockIdx.x - tok * G;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int K = D.topk;
  SelWs* W = reinterpret_cast<SelWs*>(D.sel_ws) + tok;
  __shared__ __align__(16) uint32_t hist[SEL_BINS];
  __shared__ int warp_tot[32];
  __shared__ int s_bin, s_ok, s_cnt, s_hi, s_pos, s_off;
  __shared__ long long s_above;
  __shared__ unsigned long long s_tau;
  __shared__ __align__(8) uint64_t s_bar;
  extern __shared__ __align__(16) uint8_t sw_dyn[];
  unsigned long long* cache = reinterpret_cast<unsigned long long*>(sw_dyn);   // [SW_CHUNK] keys
  unsigned long long* cand = cache + SW_CHUNK;                                  // [SW_CAND] final range

  if (tid == 0) {
    mbar_init(smem_u32(&s_bar), 1);
    fence_mbar_init();
    s_cnt = 0;
    s_hi = 0;
    s_off = 0;
  }
  for (int b = tid; b < SEL_BINS; b += SW_THREADS) hist[b] = 0;
  griddep_wait();
  int n = limit_of[tok];
  n = max(0, min(n, D.max_ctx));
  int32_t* out = topk + (size_t)tok * K;
  // a launch that returns before the barriers clears the sums the scoring kernel filled
  auto clear_hist0 = [&]() {
    if (hist0_done)
      for (int b = g * (SEL_BINS / G + 1) + tid; b < min(SEL_BINS, (g + 1) * (SEL_BINS / G + 1)); b += SW_THREADS)
        W->hist[0][b] = 0;
  };
  if (n <= K) {   // every earlier token is selected (the same for all CTAs of the token)
    griddep_launch();
    clear_hist0();
    if (g == 0)
      for (int i = tid; i < K; i += SW_THREADS) out[i] = i < n ? i : -1;
    return;
  }
  const int per = ((n + G - 1) / G + 1) & ~1;   // even: every chunk starts 16-byte aligned
  if (per > SW_CHUNK) {   // the launch sizes G so that this cannot happen; same for all CTAs of the token
    griddep_launch();
    clear_hist0();
    if (g == 0 && tid == 0) set_status(D.status, HS_ERR_BAD_ID);
    return;
  }
  const long long* s = reinterpret_cast<const long long*>(scores) + (size_t)tok * ld;
  const int lo = min(n, g * per), cnt = min(n, lo + per) - lo;
  const unsigned long long bar0 = __ldcg(&W->base);   // stored by the previous launch

  // ---- the chunk's scores by bulk copy; keys; level-0 histogram ----
  const int even = cnt & ~1;
  __syncthreads();   // barrier initialised, histogram cleared
  if (tid == 0 && even > 0) {
    const uint32_t bar = smem_u32(&s_bar);
    mbar_expect_tx(bar, (uint32_t)even * 8u);
    for (int off = 0; off < even; off += 4096)
      bulk_g2s(smem_u32(cache + off), s + lo + off, (uint32_t)min(4096, even - off) * 8u, bar);
  }
  if (tid == 0 && (cnt & 1)) cache[cnt - 1] = (unsigned long long)s[lo + cnt - 1];
  if (even > 0) mbar_wait_spin(smem_u32(&s_bar), 0, D.status);   // a timeout is recorded
  __syncthreads();
  for (int i = tid; i < cnt; i += SW_THREADS) {
    long long v = (long long)cache[i];
    if (v < 0) {
      set_status(D.status, HS_ERR_BAD_WEIGHT);
      v = 0;
    }
    const unsigned long long k = sel_key(v, lo + i);
    cache[i] = k;
    if (!hist0_done) atomicAdd(&hist[bucket_of(k, fp_keys)], 1u);
  }
  unsigned long long nbar = 0;
  bool resident = false;   // every CTA of the token has passed a barrier: all are resident
  if (!hist0_done) {
    __syncthreads();
    for (int b = tid; b < SEL_BINS; b += SW_THREADS)
      if (hist[b]) atomicAdd(&W->hist[0][b], hist[b]);
    if (!sw_barrier(&W->bar, bar0 + ++nbar * G, D.status, &s_ok)) return;
    griddep_launch();
    resident = true;
  }

  // ---- narrow the range holding the K-th largest key, level by level ----
  int need = K;
  sw_find<true>(W->hist[0], need, warp_tot, &s_bin, &s_above);
  unsigned long long base, width;
  bucket_range(s_bin, fp_keys, base, width);
  int n_range = (int)__ldcg(&W->hist[0][s_bin]);
  need -= (int)s_above;
  int level = 1;
  // keys are unique, so a range of width 1 holds one key; a level divides the width
  // by 2^12, so SW_LEVELS levels reach width 1 from the widest level-0 bucket
  while (n_range > SW_CAND && width > 1 && level < SW_LEVELS) {
    const int shift = refine_shift(width);
    __syncthreads();   // hist[s_bin] of the previous level has been read
    for (int b = tid; b < SEL_BINS; b += SW_THREADS) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < cnt; i += SW_THREADS) {
      const unsigned long long k = cache[i];
      if (in_range(k, base, width)) atomicAdd(&hist[(int)((k - base) >> shift)], 1u);
    }
    __syncthreads();
    for (int b = tid; b < SEL_BINS; b += SW_THREADS)
      if (hist[b]) atomicAdd(&W->hist[level][b], hist[b]);
    if (!sw_barrier(&W->bar, bar0 + ++nbar * G, D.status, &s_ok)) return;
    if (!resident) {
      griddep_launch();
      resident = true;
    }
    sw_find<true>(W->hist[level], need, warp_tot, &s_bin, &s_above);
    n_range = (int)__ldcg(&W->hist[level][s_bin]);
    base += (unsigned long long)s_bin << shift;
    need -= (int)s_above;
    width = 1ull << shift;
    ++level;
  }

  // ---- keys of the final range to the global list; this CTA's keys above it ----
  {
    int c_in = 0, c_hi = 0;
    for (int i = tid; i < cnt; i += SW_THREADS) {
      const unsigned long long k = cache[i];
      const bool ge = k >= base;
      c_in += ge && k - base < width;
      c_hi += ge && k - base >= width;
    }
    c_in = __reduce_add_sync(0xffffffffu, c_in);
    c_hi = __reduce_add_sync(0xffffffffu, c_hi);
    if (lane == 0) {
      atomicAdd(&s_cnt, c_in);
      atomicAdd(&s_hi, c_hi);
    }
  }
  __syncthreads();
  if (tid == 0) {
    s_pos = s_cnt ? (int)atomicAdd(&W->ncand, (uint32_t)s_cnt) : 0;
    W->above[g] = (uint32_t)s_hi;
    s_cnt = 0;
  }
  __syncthreads();
  for (int i = tid; i < cnt; i += SW_THREADS) {
    const unsigned long long k = cache[i];
    if (in_range(k, base, width)) {
      const int at = s_pos + atomicAdd(&s_cnt, 1);
      if (at < SW_CAND) W->cand[at] = k;
    }
  }
  if (!sw_barrier(&W->bar, bar0 + ++nbar * G, D.status, &s_ok)) return;
  if (!resident) griddep_launch();
  // every CTA has read the sums and appended its keys: clear a share of what
  // this launch used, and record where the next launch's barriers start
  {
    const int words = level * SEL_BINS, share = (words + G - 1) / G;
    uint32_t* sums = &W->hist[0][0];
    for (int j = g * share + tid; j < min(words, (g + 1) * share); j += SW_THREADS) sums[j] = 0;
    if (g == 0 && tid == 0) {
      W->ncand = 0;
      W->base = bar0 + nbar * G;
    }
  }

  // ---- tau: the need-th largest key of the list, found alike by every CTA ----
  const int nc = min(n_range, SW_CAND);
  for (int i = tid; i < nc; i += SW_THREADS) cand[i] = __ldcg(&W->cand[i]);
  __syncthreads();
  unsigned long long lbase = base, lwidth = width;
  int lneed = need, lcnt = nc;
  while (lcnt > 1 && lwidth > 1) {
    const int shift = refine_shift(lwidth);
    for (int b = tid; b < SEL_BINS; b += SW_THREADS) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += SW_THREADS) {
      const unsigned long long k = cand[i];
      if (in_range(k, lbase, lwidth)) atomicAdd(&hist[(int)((k - lbase) >> shift)], 1u);
    }
    __syncthreads();
    sw_find<false>(hist, lneed, warp_tot, &s_bin, &s_above);
    lcnt = (int)hist[s_bin];
    lbase += (unsigned long long)s_bin << shift;
    lneed -= (int)s_above;
    lwidth = 1ull << shift;
    __syncthreads();   // hist, s_bin and s_above read before the next level rewrites them
  }
  if (tid == 0) s_tau = lbase;
  __syncthreads();
  if (lwidth > 1)   // a single key is left in [lbase, lbase + lwidth): it is tau
    for (int i = tid; i < nc; i += SW_THREADS)
      if (in_range(cand[i], lbase, lwidth)) s_tau = cand[i];
  __syncthreads();
  const unsigned long long tau = s_tau;

  // ---- output offset: the selected keys of the CTAs before this one ----
  {
    int pre = 0;
    for (int j = tid; j < g; j += SW_THREADS) pre += (int)__ldcg(&W->above[j]);
    for (int i = tid; i < nc; i += SW_THREADS) pre += cand[i] >= tau && sel_token(cand[i]) < lo;
    pre = __reduce_add_sync(0xffffffffu, pre);
    if (lane == 0 && pre) atomicAdd(&s_off, pre);
  }
  __syncthreads();

  // ---- emit: warp w owns a contiguous range of the chunk, ballots order the lanes ----
  constexpr int NW = SW_THREADS / 32;
  const int wper = (cnt + NW - 1) / NW;
  const int wlo = min(cnt, wid * wper), whi = min(cnt, wlo + wper);
  int wcount = 0;
  for (int i = wlo + lane; i < whi; i += 32) wcount += cache[i] >= tau;
  wcount = __reduce_add_sync(0xffffffffu, wcount);
  if (lane == 0) warp_tot[wid] = wcount;
  __syncthreads();
  int wbase = s_off;
  for (int w = 0; w < wid; ++w) wbase += warp_tot[w];
  for (int i0 = wlo; i0 < whi; i0 += 32) {
    const int i = i0 + lane;
    const bool sel = i < whi && cache[i] >= tau;
    const unsigned m = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int pos = wbase + __popc(m & ((1u << lane) - 1));
      if (pos < K) out[pos] = lo + i;
      else set_status(D.status, HS_ERR_BAD_ID);
    }
    wbase += __popc(m);
  }
}

}  // namespace

hs_status launch_select_wide(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                             int32_t* d_topk, bool fp_keys, int G, bool hist0_done, cudaStream_t st) {
  if (G < 1 || G > SW_MAX_G || n < 1 || n > p->d.sel_ws_tokens || n * G > num_sms() || (hist0_done && n != 1))
    return HS_ERR_INVALID;
  if (ensure_kernel_attrs(select_wide_kernel, SW_SMEM) != HS_OK) return HS_ERR_CUDA;
  return launch_pdl(select_wide_kernel, dim3(n * G), dim3(SW_THREADS), SW_SMEM, st, 0, p->d, scores, ld, d_limit,
                    d_topk, fp_keys ? 1 : 0, G, hist0_done ? 1 : 0);
}

}  // namespace hs
