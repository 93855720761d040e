// Pieces shared by the two top-K selection kernels (one cluster per query token,
// and one wide group of CTAs per query token).
//
// Each score s of token index t is made unique and order-preserving as the key
//   key = s * 2^21 + (2^21 - 1 - t)          (s >= 0, t < 2^21)
// so the top K by (score desc, token asc) are exactly the K largest keys, and the
// K-th largest key tau selects them with the single test key >= tau.
#pragma once

#include "hs_internal.cuh"

namespace hs {

constexpr int SEL_BINS = 4096;
constexpr unsigned long long IDX_MASK = (1ull << 21) - 1;

__device__ __forceinline__ unsigned long long sel_key(long long score, int t) {
  return ((unsigned long long)score << 21) | (IDX_MASK - (unsigned long long)t);
}
__device__ __forceinline__ int sel_token(unsigned long long key) { return (int)(IDX_MASK - (key & IDX_MASK)); }

// monotone level-0 bucket of a key: exact below 64, then 64 buckets per octave
__device__ __forceinline__ int bucket1(unsigned long long v) {
  if (v < 64) return (int)v;
  int e = 63 - __clzll((long long)v);
  int m = (int)((v >> (e - 6)) & 63);
  return 64 + (e - 6) * 64 + m;
}

// Level-0 bucket of a key. Integer scores (exact int64) span many octaves: log
// buckets. Order-preserving keys of fp32 scores lie in one octave of the key space:
// their top 12 bits (sign, exponent, 3 mantissa bits) are 4,096 monotone buckets.
__device__ __forceinline__ int bucket_of(unsigned long long k, bool fp_keys) {
  return fp_keys ? (int)(k >> 41) : bucket1(k);
}

// Key range [base, base + width) of level-0 bucket b; consecutive buckets tile
// the key space without gaps.
__device__ __forceinline__ void bucket_range(int b, bool fp_keys, unsigned long long& base,
                                             unsigned long long& width) {
  if (fp_keys) {
    base = (unsigned long long)b << 41;
    width = 1ull << 41;
  } else if (b < 64) {
    base = (unsigned long long)b;
    width = 1;
  } else {
    const int e = (b - 64) / 64 + 6, m = (b - 64) % 64;
    base = (1ull << e) + ((unsigned long long)m << (e - 6));
    width = 1ull << (e - 6);
  }
}

// Shift that splits a key range of `width` (a power of two) into at most 4,096 bins.
__device__ __forceinline__ int refine_shift(unsigned long long width) {
  const int lw = 63 - __clzll((long long)width);
  return lw > 12 ? lw - 12 : 0;
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

// ---- wide selection: one group of G co-resident CTAs per query token ----------------
constexpr int SW_THREADS = 512;
constexpr int SW_CHUNK = 12288;       // keys per CTA, held in shared memory
constexpr int SW_CAND = 4096;         // keys of the final range every CTA loads to find tau
constexpr int SW_LEVELS = 6;          // histogram levels (4,096 bins each) down to single keys
constexpr int SW_MAX_G = 256;         // CTAs per query token
constexpr int SW_MIN_G = 8;
constexpr int SW_TARGET = 2048;       // keys per CTA the launch aims for
constexpr int SW_SMEM = SW_CHUNK * 8 + SW_CAND * 8 + 16;

// Per query token, in global memory. The arrival counter only grows; `base` is
// its value when a launch starts (the previous launch stores it after its last
// barrier). The histogram sums and ncand are zero between launches: each launch
// clears what it used after its last barrier.
struct SelWs {
  unsigned long long bar;             // grid-barrier arrivals, all launches
  unsigned long long base;            // bar at the start of the next launch
  uint32_t ncand;                     // keys of the final range appended to cand
  uint32_t dirty;                     // a launch gave up at a grid-wide wait; cleared by hs_get_error
  uint32_t pad[2];
  uint32_t above[SW_MAX_G];           // per CTA: its keys above the final range
  uint32_t hist[SW_LEVELS][SEL_BINS]; // per level: sum of the CTAs' histograms
  unsigned long long cand[SW_CAND];
};

// CTAs per query token the pool's selection scratch is sized for.
inline int sel_wide_min_g(int max_ctx) {
  const int g = (max_ctx + SW_CHUNK - 1) / SW_CHUNK;
  return g > SW_MIN_G ? g : SW_MIN_G;
}

// hist0_done: the level-0 histogram sums of the (single) token are already complete
// withhold: the failure-path self-test (one CTA per token never arrives at the waits)
hs_status launch_select_wide(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                             int32_t* d_topk, bool fp_keys, int G, bool hist0_done, cudaStream_t st,
                             bool withhold = false);
// one CTA per query token, no cross-CTA waits (many tokens)
hs_status launch_select_token(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                              int32_t* d_topk, bool fp_keys, cudaStream_t st);

// ---- chunked selection: many query tokens, every token's keys spread over the GPU ----
constexpr int BS_CHUNK = 8192;                                  // keys per work item (16 per thread)
constexpr int BS_CAND = 4096;                                   // most keys the threshold bucket may hold
constexpr int BS_STAGE = 2048 + BS_CAND;                        // K (<= 2048) + BS_CAND staged keys
constexpr int BS_MAX_CHUNKS = (HS_MAX_CTX + BS_CHUNK - 1) / BS_CHUNK;
constexpr int BS_MAX_TOKENS = 8192;                             // query tokens per launch (shared-memory work list)

// Per query token, in global memory. hist and done are zero between launches (the
// last histogram CTA of a token resets done, the final kernel clears hist); the
// other fields are written before they are read within a launch.
struct BselTok {
  uint32_t hist[SEL_BINS];              // level-0 histogram sums over the token's chunks
  uint32_t done;                        // chunks whose histogram is in the sums
  int32_t bin;                          // the threshold bucket: it holds the K-th largest key
  int32_t need;                         // keys to take from it (K minus the keys in higher buckets)
  int32_t crowded;                      // the bucket holds more than BS_CAND keys: full selection
  uint32_t nstage;                      // keys staged so far (buckets >= bin)
  int32_t pad[3];
  uint32_t sbase[BS_MAX_CHUNKS];        // per chunk: its first staged key
  uint32_t scount[BS_MAX_CHUNKS];       // per chunk: its staged keys, in ascending token order
  unsigned long long stage[BS_STAGE];   // the keys in buckets >= bin, chunk by chunk
};

// Three launches: level-0 histograms (the last chunk of a token finds its threshold
// bucket), staging of every key in that bucket or above, and per token tau and the
// output from the staged keys.
hs_status launch_select_batch(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                              int32_t* d_topk, bool fp_keys, cudaStream_t st);

}  // namespace hs
