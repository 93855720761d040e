// Top-K selection spread over the whole GPU: the wide selection for batches of few
// query tokens (below), the chunked selection for many tokens up to one per SM, and
// one CTA per token beyond that.
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
__device__ bool sw_barrier(SelWs* W, unsigned long long target, int32_t* status, int* s_ok) {
  unsigned long long* ctr = &W->bar;
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
          atomicExch(&W->dirty, 1u);   // this token's scratch is left half used
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

// ---- one CTA selects the top K of one token, streaming its keys from global memory ----
// Warp w owns a contiguous range of the token's keys (a multiple of 32 x ST_PER_LANE
// keys, each lane reading its keys with 16-byte loads, all in flight at once), so the
// emit pass can write its selected tokens in ascending order at a known offset.
// Passes over the keys (reads from L2): the level-0 histogram, further histogram
// levels while the range holding the K-th largest key has more than SW_CAND keys,
// the collection of that range (each warp also counts its keys above it), and the
// emit pass.

// The ST_PER_LANE keys of a lane at i (a multiple of ST_PER_LANE); keys at or beyond `hi` are 0 and
// flagged invalid (bit k of the returned mask set for a valid key k).
template <int ST_PER_LANE>
__device__ __forceinline__ uint32_t st_load_lane(const long long* s, int i, int hi,
                                                unsigned long long (&k)[ST_PER_LANE], int32_t* status) {
  longlong2 v[ST_PER_LANE / 2];
#pragma unroll
  for (int j = 0; j < ST_PER_LANE / 2; ++j)
    v[j] = i + 2 * j < hi ? __ldcg(reinterpret_cast<const longlong2*>(s + i) + j) : make_longlong2(0, 0);
  uint32_t valid = 0;
#pragma unroll
  for (int j = 0; j < ST_PER_LANE; ++j) {
    long long x = (j & 1) ? v[j >> 1].y : v[j >> 1].x;
    if (i + j < hi) {
      valid |= 1u << j;
      if (x < 0) {
        set_status(status, HS_ERR_BAD_WEIGHT);
        x = 0;
      }
    }
    k[j] = sel_key(x, i + j);
  }
  return valid;
}

// ST_PER_LANE keys per lane in flight: 8 for the many-token selection (measured best of
// 4, 8 and 16 at 32 requests x 4 tokens); the recovery
// path inside the grid-wide kernel takes 4, which keeps that kernel's registers low.
template <int ST_PER_LANE>
__device__ void select_token_cta(const long long* __restrict__ s, int n, int K, bool fp_keys, int32_t* __restrict__ out,
                                 int32_t* status, uint32_t* hist, unsigned long long* cand, int* warp_tot,
                                 int* s_small) {
  constexpr int NW = SW_THREADS / 32;
  constexpr int ST_SPAN = 32 * ST_PER_LANE;   // keys per warp step
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int* s_bin = s_small;
  int* s_cnt = s_small + 1;
  int* w_above = s_small + 2;            // [NW] keys above the final range in warp w's range
  int* w_off = w_above + NW;             // [NW] output offset of warp w
  long long* s_above = reinterpret_cast<long long*>(s_small + 2 + 2 * NW + 2);
  unsigned long long* s_tau = reinterpret_cast<unsigned long long*>(s_above + 1);
  if (n <= K) {
    for (int i = tid; i < K; i += SW_THREADS) out[i] = i < n ? i : -1;
    return;
  }
  const int wper = (n + NW * ST_SPAN - 1) / (NW * ST_SPAN) * ST_SPAN;
  const int wlo = min(n, wid * wper), whi = min(n, wlo + wper);
  unsigned long long k[ST_PER_LANE];
  // level 0
  for (int b = tid; b < SEL_BINS; b += SW_THREADS) hist[b] = 0;
  __syncthreads();
  for (int i0 = wlo; i0 < whi; i0 += ST_SPAN) {
    const uint32_t v = st_load_lane(s, i0 + lane * ST_PER_LANE, whi, k, status);
#pragma unroll
    for (int j = 0; j < ST_PER_LANE; ++j)
      if (v >> j & 1) atomicAdd(&hist[bucket_of(k[j], fp_keys)], 1u);
  }
  __syncthreads();
  int need = K;
  sw_find<false>(hist, need, warp_tot, s_bin, s_above);
  unsigned long long base, width;
  bucket_range(*s_bin, fp_keys, base, width);
  int n_range = (int)hist[*s_bin];
  need -= (int)*s_above;
  while (n_range > SW_CAND && width > 1) {
    const int shift = refine_shift(width);
    __syncthreads();
    for (int b = tid; b < SEL_BINS; b += SW_THREADS) hist[b] = 0;
    __syncthreads();
    for (int i0 = wlo; i0 < whi; i0 += ST_SPAN) {
      const uint32_t v = st_load_lane(s, i0 + lane * ST_PER_LANE, whi, k, status);
#pragma unroll
      for (int j = 0; j < ST_PER_LANE; ++j)
        if ((v >> j & 1) && in_range(k[j], base, width)) atomicAdd(&hist[(int)((k[j] - base) >> shift)], 1u);
    }
    __syncthreads();
    sw_find<false>(hist, need, warp_tot, s_bin, s_above);
    n_range = (int)hist[*s_bin];
    base += (unsigned long long)*s_bin << shift;
    need -= (int)*s_above;
    width = 1ull << shift;
  }
  // the final range to shared memory; each warp counts its keys above the range
  if (tid == 0) *s_cnt = 0;
  __syncthreads();
  int above = 0;
  for (int i0 = wlo; i0 < whi; i0 += ST_SPAN) {
    const uint32_t v = st_load_lane(s, i0 + lane * ST_PER_LANE, whi, k, status);
#pragma unroll
    for (int j = 0; j < ST_PER_LANE; ++j) {
      if (!(v >> j & 1) || k[j] < base) continue;
      if (k[j] - base < width) {
        const int at = atomicAdd(s_cnt, 1);
        if (at < SW_CAND) cand[at] = k[j];
      } else {
        ++above;
      }
    }
  }
  above = __reduce_add_sync(0xffffffffu, above);
  if (lane == 0) w_above[wid] = above;
  __syncthreads();
  // tau: the need-th largest key of the range
  const int nc = min(*s_cnt, SW_CAND);
  int lcnt = nc, lneed = need;
  while (lcnt > 1 && width > 1) {
    const int shift = refine_shift(width);
    for (int b = tid; b < SEL_BINS; b += SW_THREADS) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += SW_THREADS)
      if (in_range(cand[i], base, width)) atomicAdd(&hist[(int)((cand[i] - base) >> shift)], 1u);
    __syncthreads();
    sw_find<false>(hist, lneed, warp_tot, s_bin, s_above);
    lcnt = (int)hist[*s_bin];
    base += (unsigned long long)*s_bin << shift;
    lneed -= (int)*s_above;
    width = 1ull << shift;
    __syncthreads();
  }
  if (tid == 0) *s_tau = base;
  __syncthreads();
  if (width > 1)   // a single key is left in [base, base + width): it is tau
    for (int i = tid; i < nc; i += SW_THREADS)
      if (in_range(cand[i], base, width)) *s_tau = cand[i];
  __syncthreads();
  const unsigned long long tau = *s_tau;
  // output offsets: per warp range, its keys above the range plus its range keys >= tau
  if (tid < NW) w_off[tid] = w_above[tid];
  __syncthreads();
  for (int i = tid; i < nc; i += SW_THREADS)
    if (cand[i] >= tau) atomicAdd(&w_off[min(NW - 1, sel_token(cand[i]) / wper)], 1);
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < NW; ++w) {
      const int c = w_off[w];
      w_off[w] = acc;
      acc += c;
    }
  }
  __syncthreads();
  // emit: the lanes of a warp hold ST_PER_LANE consecutive keys each, so a lane's selected keys
  // follow those of the lanes before it
  int wbase = w_off[wid];
  for (int i0 = wlo; i0 < whi; i0 += ST_SPAN) {
    const int i = i0 + lane * ST_PER_LANE;
    const uint32_t v = st_load_lane(s, i, whi, k, status);
    int c = 0;
#pragma unroll
    for (int j = 0; j < ST_PER_LANE; ++j) c += (v >> j & 1) && k[j] >= tau;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int pos = wbase + incl - c;
#pragma unroll
    for (int j = 0; j < ST_PER_LANE; ++j)
      if ((v >> j & 1) && k[j] >= tau) {
        if (pos < K) out[pos] = i + j;
        else set_status(status, HS_ERR_BAD_ID);
        ++pos;
      }
    wbase += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Many query tokens: one CTA per token (grid-stride over tokens), no cross-CTA waits.
__global__ void __launch_bounds__(SW_THREADS, 1)
select_token_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
                    int32_t* __restrict__ topk, int n_tok, int fp_keys) {
  __shared__ __align__(16) uint32_t hist[SEL_BINS];
  __shared__ __align__(16) unsigned long long cand[SW_CAND];
  __shared__ int warp_tot[32];
  __shared__ __align__(16) int s_small[2 + 2 * (SW_THREADS / 32) + 2 + 4];
  griddep_wait();
  griddep_launch();
  for (int tok = blockIdx.x; tok < n_tok; tok += gridDim.x) {
    int n = limit_of[tok];
    n = max(0, min(n, D.max_ctx));
    select_token_cta<8>(reinterpret_cast<const long long*>(scores) + (size_t)tok * ld, n, D.topk, fp_keys != 0,
                     topk + (size_t)tok * D.topk, D.status, hist, cand, warp_tot, s_small);
    __syncthreads();
  }
}

__global__ void __launch_bounds__(SW_THREADS, 1)
select_wide_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
                   int32_t* __restrict__ topk, int fp_keys, int G, int hist0_done, int withhold) {
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
  __shared__ __align__(16) int dirty_small[2 + 2 * (SW_THREADS / 32) + 2 + 4];
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
  if (__ldcg(&W->dirty)) {
    // An earlier launch gave up at a grid-wide wait and left this token's scratch
    // half used. Until hs_get_error has reported that and cleared the scratch, the
    // token is selected by its first CTA alone, without the scratch and without waits.
    griddep_launch();
    if (g == 0)
      select_token_cta<4>(reinterpret_cast<const long long*>(scores) + (size_t)tok * ld, n, K, fp_keys != 0, out,
                       D.status, hist, cand, warp_tot, dirty_small);
    return;
  }
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
  if (withhold && g == G - 1) {
    // self-test of the failure path: this CTA never arrives at the grid-wide waits,
    // as if it could not get an SM, so the token's other CTAs give up after WAIT_NS
    griddep_launch();
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
    if (!sw_barrier(W, bar0 + ++nbar * G, D.status, &s_ok)) return;
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
    if (!sw_barrier(W, bar0 + ++nbar * G, D.status, &s_ok)) return;
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
  if (!sw_barrier(W, bar0 + ++nbar * G, D.status, &s_ok)) return;
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


// ---- chunked selection: many query tokens, each token's keys in chunks over the GPU ----
// Token t with n_t > K keys owns BS_CHUNK-key chunks first[t] .. first[t + 1] - 1 of a
// work list that every CTA builds in shared memory from the limits; a token with
// n_t <= K owns none (the final kernel writes its output).
constexpr int BS_THREADS = SW_THREADS;
constexpr int BS_PER = 8;                              // keys per 16-byte-load step of a thread
constexpr int BS_KPT = BS_CHUNK / BS_THREADS;          // keys per thread of a chunk
static_assert(BS_KPT == 2 * BS_PER, "a chunk is two load steps of every thread");
static_assert(HS_MAX_CTX % 2 == 0, "16-byte score loads stay inside a row");
constexpr int BS_EPT = (BS_STAGE + BS_THREADS - 1) / BS_THREADS;   // staged keys per thread at the end
constexpr int BS_FINAL_SMEM = BS_STAGE * 8 + 2 * (BS_MAX_CHUNKS + 1) * 4;

__device__ __forceinline__ int bs_limit(const int32_t* limit_of, int tok, int max_ctx) {
  const int n = limit_of[tok];
  return max(0, min(n, max_ctx));
}

// first[0 .. n_tok] (shared memory): exclusive prefix of the tokens' chunk counts; returns the total.
__device__ int bs_work_list(const int32_t* limit_of, int n_tok, int K, int max_ctx, int* first, int* warp_tot,
                            int* s_total) {
  int carry = 0;
  for (int base = 0; base < n_tok; base += BS_THREADS) {
    const int t = base + (int)threadIdx.x;
    int c = 0;
    if (t < n_tok) {
      const int n = bs_limit(limit_of, t, max_ctx);
      c = n > K ? (n + BS_CHUNK - 1) / BS_CHUNK : 0;
    }
    const int ex = block_excl_scan(c, warp_tot, s_total);
    if (t < n_tok) first[t] = carry + ex;
    carry += *s_total;
  }
  if (threadIdx.x == 0) first[n_tok] = carry;
  __syncthreads();
  return carry;
}

// the last t with first[t] <= w (the token that owns work item w)
__device__ __forceinline__ int bs_token_of(const int* first, int n_tok, int w) {
  int lo = 0, hi = n_tok;   // first[lo] <= w < first[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (first[mid] <= w) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Adds the CTA's histogram of nacc chunks of token B (of nch chunks) to the token's
// sums and clears it; the CTA that completes the sums finds the threshold bucket.
__device__ __noinline__ void bs_flush(BselTok* B, int nch, int nacc, int K, uint32_t* hist, int* warp_tot, int* s_bin,
                                      long long* s_above, int* s_last) {
  const int tid = threadIdx.x;
  __syncthreads();
  for (int b = tid; b < SEL_BINS; b += BS_THREADS) {
    const uint32_t h = hist[b];
    if (h) {
      atomicAdd(&B->hist[b], h);
      hist[b] = 0;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = atomicAdd(&B->done, (uint32_t)nacc) + (uint32_t)nacc == (uint32_t)nch;
  __syncthreads();
  if (*s_last) {   // every chunk's histogram of this token is in the sums
    __threadfence();
    sw_find<true>(B->hist, K, warp_tot, s_bin, s_above);
    if (tid == 0) {
      B->bin = *s_bin;
      B->need = K - (int)*s_above;
      B->crowded = __ldcg(&B->hist[*s_bin]) > (uint32_t)BS_CAND;
      B->nstage = 0;
      B->done = 0;
    }
  }
  __syncthreads();
}

// Pass 1: level-0 histograms. A CTA takes a contiguous run of chunks, sums the chunks
// of one token in shared memory and adds them to the token's global sums when the
// token changes; the CTA that completes a token's sums finds the bucket holding the
// K-th largest key and whether it is crowded.
__global__ void __launch_bounds__(BS_THREADS)
bsel_hist_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of, int n_tok,
                 int fp_keys) {
  extern __shared__ __align__(16) int bs_first[];   // [n_tok + 1]
  __shared__ __align__(16) uint32_t hist[SEL_BINS];
  __shared__ int warp_tot[32];
  __shared__ int s_total, s_bin, s_last;
  __shared__ long long s_above;
  const int tid = threadIdx.x, K = D.topk;
  BselTok* T = reinterpret_cast<BselTok*>(D.bsel);
  griddep_wait();
  griddep_launch();
  const int total = bs_work_list(limit_of, n_tok, K, D.max_ctx, bs_first, warp_tot, &s_total);
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int w0 = min(total, (int)blockIdx.x * per), w1 = min(total, w0 + per);
  for (int b = tid; b < SEL_BINS; b += BS_THREADS) hist[b] = 0;
  __syncthreads();
  int cur = -1, nacc = 0;
  for (int w = w0; w < w1; ++w) {
    const int tok = bs_token_of(bs_first, n_tok, w);
    if (tok != cur) {
      if (cur >= 0) bs_flush(T + cur, bs_first[cur + 1] - bs_first[cur], nacc, K, hist, warp_tot, &s_bin, &s_above, &s_last);
      cur = tok;
      nacc = 0;
    }
    const int c = w - bs_first[tok];
    const int n = bs_limit(limit_of, tok, D.max_ctx);
    const int lo = c * BS_CHUNK, hi = min(n, lo + BS_CHUNK);
    const long long* s = reinterpret_cast<const long long*>(scores) + (size_t)tok * ld;
    unsigned long long k[BS_PER];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lo + (2 * tid + h) * BS_PER;
      const uint32_t v = st_load_lane<BS_PER>(s, i, hi, k, D.status);
#pragma unroll
      for (int j = 0; j < BS_PER; ++j)
        if (v >> j & 1) atomicAdd(&hist[bucket_of(k[j], fp_keys != 0)], 1u);
    }
    ++nacc;
  }
  if (cur >= 0) bs_flush(T + cur, bs_first[cur + 1] - bs_first[cur], nacc, K, hist, warp_tot, &s_bin, &s_above, &s_last);
}

// Pass 2: each chunk stages its keys in the threshold bucket or above, in ascending
// token order, at a range of its token's list that it reserves with one atomic.
__global__ void __launch_bounds__(BS_THREADS)
bsel_stage_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of, int n_tok,
                  int fp_keys) {
  extern __shared__ __align__(16) int bs_first[];
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ uint32_t s_base;
  const int tid = threadIdx.x, K = D.topk;
  BselTok* T = reinterpret_cast<BselTok*>(D.bsel);
  griddep_wait();
  griddep_launch();
  const int total = bs_work_list(limit_of, n_tok, K, D.max_ctx, bs_first, warp_tot, &s_total);
  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const int tok = bs_token_of(bs_first, n_tok, w);
    BselTok* B = T + tok;
    if (__ldcg(&B->crowded)) continue;   // uniform: the final kernel selects this token in full
    const int c = w - bs_first[tok];
    const int n = bs_limit(limit_of, tok, D.max_ctx);
    const int lo = c * BS_CHUNK, hi = min(n, lo + BS_CHUNK);
    const long long* s = reinterpret_cast<const long long*>(scores) + (size_t)tok * ld;
    const int bin = __ldcg(&B->bin);
    unsigned long long k[BS_KPT], k1[BS_PER];
    // both halves' loads first, then the buckets
    const uint32_t v0 = st_load_lane<BS_PER>(s, lo + tid * BS_KPT, hi, *reinterpret_cast<unsigned long long(*)[BS_PER]>(k), D.status);
    const uint32_t v1 = st_load_lane<BS_PER>(s, lo + tid * BS_KPT + BS_PER, hi, k1, D.status);
#pragma unroll
    for (int j = 0; j < BS_PER; ++j) k[BS_PER + j] = k1[j];
    const uint32_t valid = v0 | (v1 << BS_PER);
    uint32_t take = 0;
#pragma unroll
    for (int j = 0; j < BS_KPT; ++j)
      if ((valid >> j & 1) && bucket_of(k[j], fp_keys != 0) >= bin) take |= 1u << j;
    const int ex = block_excl_scan(__popc(take), warp_tot, &s_total);
    if (tid == 0) {
      s_base = atomicAdd(&B->nstage, (uint32_t)s_total);
      B->sbase[c] = s_base;
      B->scount[c] = (uint32_t)s_total;
    }
    __syncthreads();
    uint32_t pos = s_base + (uint32_t)ex;
#pragma unroll
    for (int j = 0; j < BS_KPT; ++j)
      if (take >> j & 1) {
        if (pos < (uint32_t)BS_STAGE) B->stage[pos] = k[j];
        else set_status(D.status, HS_ERR_BAD_ID);   // not reached: a bucket this full is crowded
        ++pos;
      }
    __syncthreads();   // s_base, s_total
  }
}

// Per token (one CTA, grid-stride over tokens): tau among the staged keys, then the
// output: the staged keys >= tau in chunk order, which is ascending token order. A
// token with at most K keys gets all of them (ascending, -1 after); a crowded one is
// selected here in full. The token's sums are cleared for the next launch.
__global__ void __launch_bounds__(BS_THREADS)
bsel_final_kernel(Dev D, const int64_t* __restrict__ scores, int ld, const int32_t* __restrict__ limit_of,
                  int32_t* __restrict__ topk, int n_tok, int fp_keys) {
  extern __shared__ __align__(16) unsigned long long bs_dyn[];
  unsigned long long* st = bs_dyn;                                  // [BS_STAGE] staged keys
  int* s_pre = reinterpret_cast<int*>(st + BS_STAGE);                // [BS_MAX_CHUNKS + 1] chunk-order prefix
  int* s_sb = s_pre + BS_MAX_CHUNKS + 1;                             // [BS_MAX_CHUNKS] chunk's first staged key
  __shared__ __align__(16) uint32_t hist[SEL_BINS];
  __shared__ int warp_tot[32];
  __shared__ __align__(16) int s_small[2 + 2 * (SW_THREADS / 32) + 2 + 4];
  __shared__ int s_bin, s_total;
  __shared__ long long s_above;
  __shared__ unsigned long long s_tau;
  static_assert(BS_STAGE >= SW_CAND, "the staged-key buffer serves the full selection's candidates");
  const int tid = threadIdx.x, K = D.topk;
  BselTok* T = reinterpret_cast<BselTok*>(D.bsel);
  griddep_wait();
  griddep_launch();
  for (int tok = blockIdx.x; tok < n_tok; tok += gridDim.x) {
    const int n = bs_limit(limit_of, tok, D.max_ctx);
    int32_t* out = topk + (size_t)tok * K;
    if (n <= K) {
      for (int i = tid; i < K; i += BS_THREADS) out[i] = i < n ? i : -1;
      continue;   // uniform: no chunks, no sums
    }
    BselTok* B = T + tok;
    if (__ldcg(&B->crowded)) {   // the threshold bucket is crowded: the full selection
      select_token_cta<8>(reinterpret_cast<const long long*>(scores) + (size_t)tok * ld, n, K, fp_keys != 0, out,
                          D.status, hist, st, warp_tot, s_small);
    } else {
      const int m = min((int)__ldcg(&B->nstage), BS_STAGE), nch = (n + BS_CHUNK - 1) / BS_CHUNK;
      for (int i = tid; i < m; i += BS_THREADS) st[i] = __ldcg(&B->stage[i]);
      for (int x = tid; x < nch; x += BS_THREADS) {
        s_sb[x] = (int)__ldcg(&B->sbase[x]);
        s_pre[x + 1] = (int)__ldcg(&B->scount[x]);
      }
      __syncthreads();
      if (tid == 0) {   // at most BS_MAX_CHUNKS additions in shared memory
        s_pre[0] = 0;
        for (int x = 1; x <= nch; ++x) s_pre[x] += s_pre[x - 1];
      }
      unsigned long long base, width;
      bucket_range(__ldcg(&B->bin), fp_keys != 0, base, width);
      int lcnt = m, lneed = __ldcg(&B->need);
      __syncthreads();
      while (lcnt > 1 && width > 1) {   // narrow the bucket's range to the single key tau
        const int shift = refine_shift(width);
        for (int b = tid; b < SEL_BINS; b += BS_THREADS) hist[b] = 0;
        __syncthreads();
        for (int i = tid; i < m; i += BS_THREADS)
          if (in_range(st[i], base, width)) atomicAdd(&hist[(int)((st[i] - base) >> shift)], 1u);
        __syncthreads();
        sw_find<false>(hist, lneed, warp_tot, &s_bin, &s_above);
        lcnt = (int)hist[s_bin];
        base += (unsigned long long)s_bin << shift;
        lneed -= (int)s_above;
        width = 1ull << shift;
        __syncthreads();
      }
      if (tid == 0) s_tau = base;
      __syncthreads();
      if (width > 1)
        for (int i = tid; i < m; i += BS_THREADS)
          if (in_range(st[i], base, width)) s_tau = st[i];
      __syncthreads();
      const unsigned long long tau = s_tau;
      // virtual position v = s_pre[c] + (e - s_sb[c]) orders the staged keys by chunk
      const int mv = s_pre[nch];
      unsigned long long kv[BS_EPT];
      int cnt = 0;
#pragma unroll
      for (int j = 0; j < BS_EPT; ++j) {
        const int v = tid * BS_EPT + j;
        kv[j] = 0;
        if (v < mv) {
          int lo = 0, hi = nch;   // s_pre[lo] <= v < s_pre[hi]
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_pre[mid] <= v) lo = mid;
            else hi = mid;
          }
          const int e = s_sb[lo] + (v - s_pre[lo]);
          if (e < m) kv[j] = st[e];
        }
        cnt += kv[j] >= tau && v < mv;
      }
      int pos = block_excl_scan(cnt, warp_tot, &s_total);
#pragma unroll
      for (int j = 0; j < BS_EPT; ++j)
        if (tid * BS_EPT + j < mv && kv[j] >= tau) {
          if (pos < K) out[pos] = sel_token(kv[j]);
          ++pos;
        }
      if (tid == 0 && s_total != K) set_status(D.status, HS_ERR_BAD_ID);   // exactly K keys are >= tau
    }
    for (int b = tid; b < SEL_BINS; b += BS_THREADS) B->hist[b] = 0;
    __syncthreads();
  }
}

}  // namespace

hs_status launch_select_token(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                              int32_t* d_topk, bool fp_keys, cudaStream_t st) {
  if (n < 1) return HS_ERR_INVALID;
  const int grid = n < num_sms() ? n : num_sms();
  return launch_pdl(select_token_kernel, dim3(grid), dim3(SW_THREADS), 0, st, 0, p->d, scores, ld, d_limit, d_topk,
                    n, fp_keys ? 1 : 0);
}

hs_status launch_select_batch(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                              int32_t* d_topk, bool fp_keys, cudaStream_t st) {
  if (n < 1 || n > p->d.bsel_tokens || !p->d.bsel) return HS_ERR_INVALID;
  const int smem = (n + 1) * (int)sizeof(int);
  constexpr int smem_max = (BS_MAX_TOKENS + 1) * (int)sizeof(int);
  if (ensure_kernel_attrs(bsel_hist_kernel, smem_max) != HS_OK || ensure_kernel_attrs(bsel_stage_kernel, smem_max) != HS_OK ||
      ensure_kernel_attrs(bsel_final_kernel, BS_FINAL_SMEM) != HS_OK)
    return HS_ERR_CUDA;
  // two CTAs per SM for the staging pass (its registers), three for the lighter
  // histogram pass: more chunks in flight per SM
  const int grid = 2 * num_sms(), fk = fp_keys ? 1 : 0;
  hs_status s = launch_pdl(bsel_hist_kernel, dim3(3 * num_sms()), dim3(BS_THREADS), smem, st, 0, p->d, scores, ld,
                           d_limit, n, fk);
  if (s == HS_OK)
    s = launch_pdl(bsel_stage_kernel, dim3(grid), dim3(BS_THREADS), smem, st, 0, p->d, scores, ld, d_limit, n, fk);
  if (s == HS_OK)
    s = launch_pdl(bsel_final_kernel, dim3(n < 2 * num_sms() ? n : 2 * num_sms()), dim3(BS_THREADS), BS_FINAL_SMEM, st,
                   0, p->d, scores, ld, d_limit, d_topk, n, fk);
  if (s != HS_OK)   // a launch after the first failed: its sums must not reach the next call
    cudaMemsetAsync(p->d.bsel, 0, (size_t)p->d.bsel_tokens * sizeof(BselTok), st);
  return s;
}

hs_status launch_select_wide(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                             int32_t* d_topk, bool fp_keys, int G, bool hist0_done, cudaStream_t st, bool withhold) {
  if (G < 2 || G > SW_MAX_G || n < 1 || n > p->d.sel_ws_tokens || n * G > num_sms() || (hist0_done && n != 1))
    return HS_ERR_INVALID;
  if (ensure_kernel_attrs(select_wide_kernel, SW_SMEM) != HS_OK) return HS_ERR_CUDA;
  return launch_pdl(select_wide_kernel, dim3(n * G), dim3(SW_THREADS), SW_SMEM, st, 0, p->d, scores, ld, d_limit,
                    d_topk, fp_keys ? 1 : 0, G, hist0_done ? 1 : 0, withhold ? 1 : 0);
}

}  // namespace hs
