// Sparse MLA decode attention over the resolved rows, MQA form.
//
// "Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse" (vLLM blog Part 2),
// footnote 1: each query reads its 2,048 selected 656-byte FP8 rows; QK runs over
// 576 dims and PV over 512; every row serves all 64 heads (section "PCP: split
// tokens, not heads"), which is what puts sparse MLA near the compute ridge.
//
// One CTA (16 warps) per (query token, group of HPC heads, block of 128 selected
// rows); the row-block CTAs of one (token, head group) form a thread-block
// cluster. HPC is 64 for large batches and 16 or 32 when few query tokens would
// leave most SMs idle: the head groups then run as independent clusters, which
// spreads one token over more SMs and shortens every per-CTA phase after the
// gather (each head group gathers the same rows; the repeats hit L2).
//  * every thread loads ~10 of the block's 16-byte row chunks at once, gathered by
//    HMA row id (one stride for resident and hot rows; chunks dealt by row_piece so
//    that the stores of one shared-memory cycle hit distinct banks), and puts each chunk in
//    place: the FP8 latent widened to bf16 by a bit shuffle that is exact up to
//    the constant factor 2^-120 (normal and subnormal e4m3 alike), the fp32 group
//    scales to a small table, the bf16 rope unchanged; the 128 x 576 bf16 tile
//    (128-byte swizzle) is the K-major A operand of QK and the MN-major A
//    operand of PV; the bf16 query is the K-major B operand unchanged;
//  * QK on tcgen05 into five TMEM accumulators (four 128-dim latent groups and
//    the rope), so each row's per-group scales (x 2^120) are applied in fp32 when
//    the scores are read back: s = sum_g scale_g * S_g + S_rope;
//  * softmax from TMEM: each thread owns one row and HPC/4 heads; per-head max
//    and sum over rows use a warp transpose-reduction and shared memory;
//  * PV on tcgen05 per latent group g with P_g = p * scale_g * 2^120 (bf16),
//    so the unscaled FP8 values serve as V;
//  * split merge with one cluster barrier: while PV runs, each CTA writes its
//    per-head (max, sum) to the token's merge record; after PV it writes its
//    partial output, normalised by its own sum and rounded to fp16, to a
//    per-token merge buffer (both stay in L2). After the barrier each CTA turns
//    the (max, sum) of all splits into log-sum-exp weights (a 16-lane group per
//    head), sums one slice of the 512 output dims over the splits in fp32,
//    transposes it through shared memory and writes it as bf16 in 16-byte pieces.
// Per-group scales must stay below 256 (so scale * 2^120 fits fp32 and bf16).
#include "hs_internal.cuh"

namespace hs {

constexpr int AT_THREADS = 512;
constexpr int AT_KV_COL = ATTN_ROWS * 128;       // 16 KB: one 64-dim bf16 atom column of the tile
constexpr int AT_OFF_KV = 0;
constexpr int AT_OFF_Q = 9 * AT_KV_COL;          // 144 KB; after QK the query region holds P_0..P_3
constexpr int AT_MISC = 6144;
constexpr int AT_CHUNKS = ATTN_ROWS * ROW_CHUNKS;        // 5,248 16-byte chunks per block
constexpr int AT_CPT = (AT_CHUNKS + AT_THREADS - 1) / AT_THREADS;   // 11 per thread
constexpr float LOG2E = 1.4426950408889634f;
constexpr float TWO_POW_120 = 1.329227995784916e36f;

// Shared-memory plan for HPC heads per CTA.
template <int HPC>
struct AtPlan {
  static constexpr int Q_COL = HPC * 128;                 // one 64-dim atom column of Q [HPC][576]
  static constexpr int P_G = 2 * HPC * 128;               // one P_g [HPC heads][128 rows] bf16
  static constexpr int OFF_MISC = AT_OFF_Q + 9 * Q_COL;
  // Up to 32 heads the splits merge in shared memory: each CTA receives, by
  // asynchronous remote stores, every split's per-head (max, sum) and the fp16
  // partials of its own slice of the output dims. At 64 heads that does not fit;
  // the merge goes through an L2-resident buffer instead.
  static constexpr bool DSM = HPC <= 32;
  static constexpr int RECV_DIMS = HPC == 16 ? 600 : 512;         // splits x slice dims it can receive
  static constexpr int RECV = DSM ? RECV_DIMS * HPC * 2 : 0;      // [split][slice dim][HPC] fp16
  static constexpr int STATS = DSM ? MAX_SPLITS * HPC * 8 : 0;    // [split][HPC] (max, sum)
  static constexpr int OFF_RECV = OFF_MISC + AT_MISC;
  static constexpr int OFF_STATS = OFF_RECV + RECV;
  static constexpr int SMEM = OFF_STATS + STATS + 1024;
  static constexpr int HW = HPC / 4;                      // heads per warp in the softmax
  static_assert(4 * P_G <= 9 * Q_COL, "P_0..P_3 fit in the query region");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(HPC * 512 * 4 + MAX_SPLITS * HPC * 4 <= 9 * AT_KV_COL, "merge scratch fits in the KV region");
};

// Four e4m3 bytes -> four bf16 values times 2^-120 (exact for every finite code):
// the e4m3 exponent/mantissa bits land on the bf16 exponent/mantissa fields.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4_scaled(uint32_t w) {
  const uint32_t lo = __byte_perm(w, 0u, 0x4140);   // bytes b0, b1 -> halves (0x00b0, 0x00b1)
  const uint32_t hi = __byte_perm(w, 0u, 0x4342);   // bytes b2, b3
  const uint32_t a = ((lo & 0x00800080u) << 8) | ((lo & 0x007F007Fu) << 4);
  const uint32_t b = ((hi & 0x00800080u) << 8) | ((hi & 0x007F007Fu) << 4);
  return make_uint2(a, b);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float x, float y) {
  __nv_bfloat162 v = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Reduces each of the HW values over the 32 lanes of the warp; afterwards lane l
// holds the reduction of v[l % HW]. The first log2(HW) steps exchange half of the
// values with the partner lane (a transpose), the rest are plain butterflies.
template <int HW, bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[HW]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = HW / 2; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = hi ? v[i] : v[i + o];
      const float keep = hi ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
#pragma unroll
  for (int o = HW; o < 32; o <<= 1) {
    const float other = __shfl_xor_sync(0xffffffffu, v[0], o);
    v[0] = MAX ? fmaxf(v[0], other) : v[0] + other;
  }
  return v[0];
}


template <int HPC>
__global__ void __launch_bounds__(AT_THREADS, 1)
attention_kernel(Dev D, int layer, const uint16_t* __restrict__ q, const int32_t* __restrict__ row_ids,
                 float scale_log2, uint16_t* __restrict__ out, float* __restrict__ lse_out, int settled) {
  using PL = AtPlan<HPC>;
  constexpr int HW = PL::HW;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = smem + AT_OFF_KV;
  uint8_t* Qs = smem + AT_OFF_Q;
  uint8_t* Ps = smem + AT_OFF_Q;                                             // P_g after QK
  int32_t* ids = reinterpret_cast<int32_t*>(smem + PL::OFF_MISC);           // [128]
  float4* scl = reinterpret_cast<float4*>(ids + ATTN_ROWS);                  // [128] group scales
  float* red = reinterpret_cast<float*>(scl + ATTN_ROWS);                    // [4][HPC]
  float* mfin = red + 4 * HPC;                                               // [HPC] this split's max (log2 units)
  float* lfin = mfin + HPC;                                                  // [HPC] this split's sum
  float* wmine = lfin + HPC;                                                 // [HPC] weight of this split
  float* gstat = wmine + HPC;                                                // [HPC] lse
  uint64_t* bar = reinterpret_cast<uint64_t*>(gstat + HPC);                  // [4] QK, PV, stats in, partials in
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 4);
  __half* recv = reinterpret_cast<__half*>(smem + PL::OFF_RECV);
  float* rstats = reinterpret_cast<float*>(smem + PL::OFF_STATS);

  // the row splits of a (token, head group) are the x extent of the grid, one cluster
  // when there are several; a single split (top-K <= 128) is launched without a cluster
  const uint32_t split = blockIdx.x;
  const uint32_t n_splits = gridDim.x;
  const int H = D.n_heads, K = D.topk;
  const int n_hgrp = H / HPC;
  const int tok = blockIdx.y / n_hgrp, hgrp = blockIdx.y - tok * n_hgrp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* kv = D.kv[layer];
  const long long max_row = (long long)D.num_pages * PAGE;

  if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
  // this CTA's slice of the 512 output dims in the split merge
  const int slice = ((512 + (int)n_splits - 1) / (int)n_splits + 7) & ~7;
  const int d_lo = min(512, (int)split * slice), d_hi = min(512, d_lo + slice);
  const int nd = d_hi - d_lo;
  if (tid == 0) {
    mbar_init(smem_u32(bar), 5);       // one arrival per QK accumulator
    mbar_init(smem_u32(bar + 1), 4);   // one arrival per PV group
    if constexpr (PL::DSM) {
      mbar_init(smem_u32(bar + 2), 1);
      mbar_init(smem_u32(bar + 3), 1);
      // the bytes every split will store here: (max, sum) of all heads, partials of the slice
      mbar_expect_tx(smem_u32(bar + 2), n_splits * HPC * 8);
      mbar_expect_tx(smem_u32(bar + 3), n_splits * nd * HPC * 2);
    }
    fence_mbar_init();
  }
  if (PL::DSM && n_splits > 1) cluster_arrive_relaxed();   // this CTA has started; its barriers are initialised
  // q is an input of the call, final before the preceding kernel started: it is
  // loaded while that kernel finishes. Settled: the row ids and the rows were
  // written before it too (an earlier layer of the same selection), so they are
  // gathered meanwhile as well, through L2.
  const uint16_t* qt = q + ((size_t)tok * H + (size_t)hgrp * HPC) * QK;
  constexpr int QPT = (HPC * 72 + AT_THREADS - 1) / AT_THREADS;
  uint4 qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int c = tid + k * AT_THREADS;
    qv[k] = c < HPC * 72 ? __ldg(reinterpret_cast<const uint4*>(qt) + c) : make_uint4(0, 0, 0, 0);
  }
  if (!settled) {
    griddep_wait();
    griddep_launch();
  }
  if (tid < ATTN_ROWS) {
    const int k = (int)split * ATTN_ROWS + tid;
    const int32_t* src = row_ids + (size_t)tok * K + k;
    int id = k < K ? (settled ? __ldcg(src) : *src) : -1;
    if (id >= max_row) { set_status(D.status, HS_ERR_BAD_ID); id = -1; }
    ids[tid] = id;
  }
  // ---- Q: this head group's [HPC, 576] bf16, 72 chunks of 8 per head (loaded above) ----
  __syncthreads();   // ids ready
  // ---- all row chunks in flight at once: chunk c = row * 41 + part ----
  uint4 rc[AT_CPT];
#pragma unroll
  for (int k = 0; k < AT_CPT; ++k) {
    const int c = tid + k * AT_THREADS;
    rc[k] = make_uint4(0, 0, 0, 0);
    if (c < AT_CHUNKS) {
      int r, part;
      row_piece(c, r, part);
      const int id = ids[r];
      if (id >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(kv + (size_t)id * ROW) + part;
        rc[k] = settled ? __ldcg(src) : __ldg(src);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int c = tid + k * AT_THREADS;
    if (c < HPC * 72) {
      const int h = c / 72, ch = c - h * 72;
      *reinterpret_cast<uint4*>(Qs + (ch >> 3) * PL::Q_COL + sw128_chunk(h, ch & 7)) = qv[k];
    }
  }
#pragma unroll
  for (int k = 0; k < AT_CPT; ++k) {
    const int c = tid + k * AT_THREADS;
    if (c < AT_CHUNKS) {
      int r, part;
      row_piece(c, r, part);
      const uint4 v = rc[k];
      if (part < 32) {            // 16 latent bytes = dims 16 part .. 16 part + 15
        const uint2 a = e4m3x4_to_bf16x4_scaled(v.x), b = e4m3x4_to_bf16x4_scaled(v.y);
        const uint2 cc = e4m3x4_to_bf16x4_scaled(v.z), d = e4m3x4_to_bf16x4_scaled(v.w);
        uint8_t* col = KV + (part >> 2) * AT_KV_COL;
        const int chunk = (part & 3) * 2;
        *reinterpret_cast<uint4*>(col + sw128_chunk(r, chunk)) = make_uint4(a.x, a.y, b.x, b.y);
        *reinterpret_cast<uint4*>(col + sw128_chunk(r, chunk + 1)) = make_uint4(cc.x, cc.y, d.x, d.y);
      } else if (part == 32) {    // the four fp32 group scales
        scl[r] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
      } else {                    // 8 bf16 rope values
        *reinterpret_cast<uint4*>(KV + 8 * AT_KV_COL + sw128_chunk(r, part - 33)) = v;
      }
    }
  }
  if (settled) {
    griddep_wait();
    griddep_launch();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;

  // ---- S_g^T = KV_g . Q_g^T (g = 0..3 latent groups, 4 = rope): M = 128 rows, N = HPC ----
  // One issuing thread per accumulator (warp g, lane 0): at small N the MMAs are
  // short and the issue itself is the cost, so five threads issue side by side.
  if (lane == 0 && warp < 5) {
    const int g = warp;
    const uint32_t idesc = idesc_f16(128, HPC, false, false, true);
    const uint32_t a0 = smem_u32(KV), b0 = smem_u32(Qs);
    const int k0 = g * 8, k1 = g < 4 ? k0 + 8 : 36;   // 8 k-steps of 16 dims per group, 4 for the rope
#pragma unroll 4
    for (int kk = k0; kk < k1; ++kk) {
      const uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * AT_KV_COL + (kk & 3) * 32, 16, 1024);
      const uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * PL::Q_COL + (kk & 3) * 32, 16, 1024);
      umma_f16(tmem + g * 64, ad, bd, idesc, kk != k0);
    }
    umma_commit(smem_u32(bar));
  }
  ok &= mbar_wait(smem_u32(bar), 0, D.status);
  tc_fence_after();

  // ---- softmax over the 128 rows, per head: warp (row quadrant, HW-head quarter) ----
  const int quad = warp & 3, sub = warp >> 2;
  const int row = quad * 32 + lane;
  const bool valid = ids[row] >= 0;
  const float4 sc4 = scl[row];
  const float sg[4] = {sc4.x * TWO_POW_120, sc4.y * TWO_POW_120, sc4.z * TWO_POW_120, sc4.w * TWO_POW_120};
  float z[HW];
  {
    const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(sub * HW);
    // rope part and the four groups in one wave (two waves at 16 heads per warp, for registers)
    constexpr int WAVE = HW >= 16 ? 2 : 4;
    uint32_t r[WAVE + 1][HW];
    tmem_ld_cols<HW>(ta + 256, r[WAVE]);
#pragma unroll
    for (int g = 0; g < WAVE; ++g) tmem_ld_cols<HW>(ta + g * 64, r[g]);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < HW; ++i) {
      float acc = __uint_as_float(r[WAVE][i]);
#pragma unroll
      for (int g = 0; g < WAVE; ++g) acc = fmaf(__uint_as_float(r[g][i]), sg[g], acc);
      z[i] = acc;
    }
    if constexpr (WAVE < 4) {
#pragma unroll
      for (int g = WAVE; g < 4; ++g) tmem_ld_cols<HW>(ta + g * 64, r[g - WAVE]);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < HW; ++i)
#pragma unroll
        for (int g = WAVE; g < 4; ++g) z[i] = fmaf(__uint_as_float(r[g - WAVE][i]), sg[g], z[i]);
    }
#pragma unroll
    for (int i = 0; i < HW; ++i) z[i] = valid ? z[i] * scale_log2 : -INFINITY;
    float t[HW];
#pragma unroll
    for (int i = 0; i < HW; ++i) t[i] = z[i];
    const float m = warp_transpose_reduce<HW, true>(t);
    if (lane < HW) red[quad * HPC + sub * HW + lane] = m;
  }
  __syncthreads();
  if (tid < HPC) mfin[tid] = fmaxf(fmaxf(red[tid], red[HPC + tid]), fmaxf(red[2 * HPC + tid], red[3 * HPC + tid]));
  __syncthreads();
  {
    float t[HW];
#pragma unroll
    for (int i = 0; i < HW; ++i) {
      const float m = mfin[sub * HW + i];
      const float p = (m == -INFINITY || z[i] == -INFINITY) ? 0.f : exp2f(z[i] - m);
      z[i] = p;
      t[i] = p;
    }
    const float l = warp_transpose_reduce<HW, false>(t);
    if (lane < HW) red[quad * HPC + sub * HW + lane] = l;
    // P_g = p * scale_g * 2^120 (bf16), the B operand of group g's PV. At 64 heads
    // it is MN-major, P_g^T[row][head] with one 128-byte line per row (16-byte
    // stores); below that a line would be shorter than the swizzle atom, so it is
    // K-major, P_g[head][row], written element by element.
    if constexpr (HPC == 64) {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
#pragma unroll
        for (int c = 0; c < HW / 8; ++c) {
          const float* zz = z + 8 * c;
          *reinterpret_cast<uint4*>(Ps + g * PL::P_G + sw128_chunk(row, sub * (HW / 8) + c)) =
              make_uint4(pack_bf16x2(zz[0] * sg[g], zz[1] * sg[g]), pack_bf16x2(zz[2] * sg[g], zz[3] * sg[g]),
                         pack_bf16x2(zz[4] * sg[g], zz[5] * sg[g]), pack_bf16x2(zz[6] * sg[g], zz[7] * sg[g]));
        }
      }
    } else {
      uint16_t* pbase = reinterpret_cast<uint16_t*>(Ps + (row >> 6) * (HPC * 128));
#pragma unroll
      for (int g = 0; g < 4; ++g) {
#pragma unroll
        for (int i = 0; i < HW; ++i) {
          const int h = sub * HW + i;
          pbase[(g * PL::P_G + sw128_off(h, row & 63)) >> 1] = __bfloat16_as_ushort(__float2bfloat16_rn(z[i] * sg[g]));
        }
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();   // every S read: the accumulators may be overwritten by PV
  tc_fence_after();

  // ---- O_g^T = V_g^T . P_g^T : M = 128 latent dims, N = HPC, K = 128 rows (warp g issues) ----
  if (lane == 0 && warp < 4) {
    const int g = warp;
    constexpr bool P_MN = HPC == 64;
    const uint32_t idesc = idesc_f16(128, HPC, true, P_MN, true);
    const uint32_t kv0 = smem_u32(KV), p0 = smem_u32(Ps);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t ad = smem_desc_sw128(kv0 + (2 * g) * AT_KV_COL + kk * 2048, AT_KV_COL, 1024);
      const uint64_t bd =
          P_MN ? smem_desc_sw128(p0 + g * PL::P_G + kk * 2048, PL::P_G, 1024)
               : smem_desc_sw128(p0 + g * PL::P_G + (kk >> 2) * (HPC * 128) + (kk & 3) * 32, 16, 1024);
      umma_f16(tmem + g * 64, ad, bd, idesc, kk > 0);
    }
    umma_commit(smem_u32(bar + 1));
  }
  if (n_splits == 1) {
    // ---- one split holds every selected row: its output, normalised by its own sum,
    //      is final; no merge and no cluster instruction (the launch has no cluster) ----
    if (tid < HPC) {
      const float l = red[tid] + red[HPC + tid] + red[2 * HPC + tid] + red[3 * HPC + tid];
      lfin[tid] = l;
      gstat[tid] = l > 0.f ? (mfin[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    ok &= mbar_wait(smem_u32(bar + 1), 0, D.status);
    tc_fence_after();
    __syncthreads();   // lfin
    {
      const int g = sub;
      const int dim = g * 128 + quad * 32 + lane;   // warp (row quadrant, group g): one dim per lane
      constexpr int CW = HPC < 32 ? HPC : 32;       // columns per TMEM read
      uint16_t* o = out + ((size_t)tok * H + (size_t)hgrp * HPC) * 512 + dim;
#pragma unroll
      for (int h0 = 0; h0 < HPC; h0 += CW) {
        uint32_t r[CW];
        tmem_ld_cols<CW>(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * 64 + h0), r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const float l = lfin[h0 + j];
          o[(size_t)(h0 + j) * 512] = __bfloat16_as_ushort(__float2bfloat16_rn(l > 0.f ? __uint_as_float(r[j]) / l : 0.f));
        }
      }
    }
    if (lse_out && tid < HPC) lse_out[(size_t)tok * H + (size_t)hgrp * HPC + tid] = gstat[tid];
  } else if constexpr (PL::DSM) {
    // while PV runs: this split's per-head (max, sum) into every CTA of the cluster
    cluster_wait_acquire();   // every CTA has started and initialised its barriers
    if (tid >= 128 && tid < 128 + HPC) {
      const int h = tid - 128;
      const float l = red[h] + red[HPC + h] + red[2 * HPC + h] + red[3 * HPC + h];
      lfin[h] = l;
      const uint32_t a = smem_u32(rstats + ((int)split * HPC + h) * 2), rb = smem_u32(bar + 2);
      for (uint32_t d = 0; d < n_splits; ++d) st_async_v2f(mapa(a, d), mfin[h], l, mapa(rb, d));
    }
    ok &= mbar_wait(smem_u32(bar + 1), 0, D.status);
    tc_fence_after();
    __syncthreads();   // lfin
    // ---- the split's partial O, normalised by its own sum, in fp16 straight into the
    //      shared memory of the CTA that owns the dims: warp (row quadrant, group g) ----
    {
      const int g = sub;
      const int dim = g * 128 + quad * 32 + lane;
      const int owner = dim / slice;
      const uint32_t dst = mapa(smem_u32(recv + ((size_t)split * slice + (dim - owner * slice)) * HPC), owner);
      const uint32_t rb = mapa(smem_u32(bar + 3), owner);
      uint32_t r[HPC];
      tmem_ld_cols<HPC>(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * 64), r);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < HPC / 8; ++c) {
        uint32_t hv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = c * 8 + 2 * i;
          const float i0 = lfin[h] > 0.f ? 1.f / lfin[h] : 0.f, i1 = lfin[h + 1] > 0.f ? 1.f / lfin[h + 1] : 0.f;
          __half2 h2 = __floats2half2_rn(__uint_as_float(r[h]) * i0, __uint_as_float(r[h + 1]) * i1);
          hv[i] = *reinterpret_cast<uint32_t*>(&h2);
        }
        st_async_v4(dst + c * 16, make_uint4(hv[0], hv[1], hv[2], hv[3]), rb);
      }
    }
    // ---- weights of the splits per head (16-lane group per head), from this CTA's copy ----
    float* wts = reinterpret_cast<float*>(KV);            // [MAX_SPLITS][HPC]; the KV tile is no longer read
    float* tr = wts + MAX_SPLITS * HPC;                    // [HPC][slice] fp32 transpose
    ok &= mbar_wait(smem_u32(bar + 2), 0, D.status);
    if (tid < MAX_SPLITS * HPC) {                          // whole warps (16 x HPC is a multiple of 32)
      const int h = tid >> 4, sp = tid & 15;
      const float2 ml = sp < (int)n_splits ? *reinterpret_cast<const float2*>(rstats + (sp * HPC + h) * 2)
                                           : make_float2(-INFINITY, 0.f);
      float M = ml.x;
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float e = ml.x == -INFINITY ? 0.f : ml.y * exp2f(ml.x - M);
      float L = e;
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      wts[sp * HPC + h] = L > 0.f ? e / L : 0.f;
      if (sp == 0) gstat[h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    ok &= mbar_wait(smem_u32(bar + 3), 0, D.status);   // every split's partials of this slice
    for (int e = tid; e < nd * (HPC / 8); e += AT_THREADS) {
      const int dd = e / (HPC / 8), h8 = e - dd * (HPC / 8);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int sp = 0; sp < (int)n_splits; ++sp) {
        const uint4 v = *reinterpret_cast<const uint4*>(recv + ((size_t)sp * slice + dd) * HPC + h8 * 8);
        const float4 w0 = *reinterpret_cast<const float4*>(wts + sp * HPC + h8 * 8);
        const float4 w1 = *reinterpret_cast<const float4*>(wts + sp * HPC + h8 * 8 + 4);
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x[k]));
          acc[2 * k] = fmaf(w[2 * k], f.x, acc[2 * k]);
          acc[2 * k + 1] = fmaf(w[2 * k + 1], f.y, acc[2 * k + 1]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) tr[(h8 * 8 + j) * slice + dd] = acc[j];
    }
    __syncthreads();
    const int nc = nd >> 3;
    for (int e = tid; e < HPC * nc; e += AT_THREADS) {
      const int h = e / nc, c = e - h * nc;
      const float* src = tr + h * slice + c * 8;
      *reinterpret_cast<uint4*>(out + ((size_t)tok * H + (size_t)hgrp * HPC + h) * 512 + d_lo + c * 8) =
          make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]), pack_bf16x2(src[4], src[5]),
                     pack_bf16x2(src[6], src[7]));
    }
    if (split == 0 && lse_out && tid < HPC) lse_out[(size_t)tok * H + (size_t)hgrp * HPC + tid] = gstat[tid];
  } else {
    // while PV runs: this split's per-head (max, sum) to the token's merge record
    float2* stats = D.o_stats + (size_t)tok * MAX_SPLITS * 64;          // [split][64 heads]
    if (tid >= 128 && tid < 128 + HPC) {
      const int h = tid - 128;
      const float l = red[h] + red[HPC + h] + red[2 * HPC + h] + red[3 * HPC + h];
      lfin[h] = l;
      stats[(size_t)split * 64 + hgrp * HPC + h] = make_float2(mfin[h], l);
    }
    ok &= mbar_wait(smem_u32(bar + 1), 0, D.status);
    tc_fence_after();
    __syncthreads();   // lfin

    // ---- the split's partial O, normalised by its own sum, in fp16 to the merge buffer ----
    // layout per (token, head group): [split][dim][HPC]; warp (row quadrant, group g)
    __half* part = D.o_part + (size_t)tok * MAX_SPLITS * 512 * 64 + (size_t)hgrp * MAX_SPLITS * 512 * HPC;
    {
      const int g = sub;
      const int dim = g * 128 + quad * 32 + lane;
      constexpr int CW = HPC < 32 ? HPC : 32;   // columns per TMEM read
      uint4* dst = reinterpret_cast<uint4*>(part + ((size_t)split * 512 + dim) * HPC);
#pragma unroll
      for (int h0 = 0; h0 < HPC; h0 += CW) {
        uint32_t r[CW];
        tmem_ld_cols<CW>(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * 64 + h0), r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < CW / 8; ++c) {
          uint32_t hv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int h = h0 + c * 8 + 2 * i;
            const float i0 = lfin[h] > 0.f ? 1.f / lfin[h] : 0.f, i1 = lfin[h + 1] > 0.f ? 1.f / lfin[h + 1] : 0.f;
            __half2 h2 = __floats2half2_rn(__uint_as_float(r[h - h0]) * i0, __uint_as_float(r[h - h0 + 1]) * i1);
            hv[i] = *reinterpret_cast<uint32_t*>(&h2);
          }
          dst[(h0 >> 3) + c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        }
      }
    }
    // one cluster barrier: every split's (max, sum) and partial are written (cluster scope)
    tc_fence_before();
    cluster_arrive_release();
    cluster_wait_acquire();

    // ---- this CTA's slice of the 512 dims: the partials are loaded first, so their
    //      round trip to L2 overlaps the one for the (max, sum) of the splits ----
    float* wts = reinterpret_cast<float*>(KV);            // [MAX_SPLITS][HPC]; the KV tile is no longer read
    float* tr = wts + MAX_SPLITS * HPC;                    // [HPC][slice] fp32 transpose
    {
      // items (dim, 8 heads); a thread's first item is loaded before the weights are known
      const int n_items = nd * (HPC / 8);
      uint4 v[MAX_SPLITS];
      auto load_item = [&](int e) {
        const int dd = e / (HPC / 8), h8 = e - dd * (HPC / 8);
#pragma unroll
        for (int sp = 0; sp < MAX_SPLITS; ++sp)   // coherent loads: written during this kernel
          v[sp] = sp < (int)n_splits ? ld_cg_v4(part + ((size_t)sp * 512 + d_lo + dd) * HPC + h8 * 8)
                                     : make_uint4(0, 0, 0, 0);
      };
      if (tid < n_items) load_item(tid);
      // weights of the splits per head: a 16-lane group per head, one lane per split
      for (int t0 = 0; t0 < MAX_SPLITS * HPC; t0 += AT_THREADS) {
        const int t = t0 + tid;
        if (t0 + (tid & ~31) < MAX_SPLITS * HPC) {           // whole warps only: shuffles below
          const int h = t >> 4, sp = t & 15;
          const float2 ml = sp < (int)n_splits ? ld_cg_f2(stats + (size_t)sp * 64 + hgrp * HPC + h)
                                               : make_float2(-INFINITY, 0.f);
          float M = ml.x;
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          const float e = ml.x == -INFINITY ? 0.f : ml.y * exp2f(ml.x - M);
          float L = e;
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
          wts[sp * HPC + h] = L > 0.f ? e / L : 0.f;
          if (sp == 0) gstat[h] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
        }
      }
      __syncthreads();
      for (int e = tid; e < n_items; e += AT_THREADS) {
        if (e != tid) load_item(e);
        const int dd = e / (HPC / 8), h8 = e - dd * (HPC / 8);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int sp = 0; sp < MAX_SPLITS; ++sp) {
          const float4 w0 = *reinterpret_cast<const float4*>(wts + sp * HPC + h8 * 8);
          const float4 w1 = *reinterpret_cast<const float4*>(wts + sp * HPC + h8 * 8 + 4);
          const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          const uint32_t x[4] = {v[sp].x, v[sp].y, v[sp].z, v[sp].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x[k]));
            acc[2 * k] = fmaf(w[2 * k], f.x, acc[2 * k]);
            acc[2 * k + 1] = fmaf(w[2 * k + 1], f.y, acc[2 * k + 1]);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) tr[(h8 * 8 + j) * slice + dd] = acc[j];
      }
    }
    {
      __syncthreads();
      const int nc = nd >> 3;
      for (int e = tid; e < HPC * nc; e += AT_THREADS) {
        const int h = e / nc, c = e - h * nc;
        const float* src = tr + h * slice + c * 8;
        *reinterpret_cast<uint4*>(out + ((size_t)tok * H + (size_t)hgrp * HPC + h) * 512 + d_lo + c * 8) =
            make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]), pack_bf16x2(src[4], src[5]),
                       pack_bf16x2(src[6], src[7]));
      }
      if (split == 0 && lse_out && tid < HPC) lse_out[(size_t)tok * H + (size_t)hgrp * HPC + tid] = gstat[tid];
    }
  }
  (void)ok;
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int HPC>
static hs_status launch_attention_hpc(hs_pool* p, int layer, int n, int n_splits, const uint16_t* d_q,
                                      const int32_t* d_rows, float scale_log2, uint16_t* d_out, float* d_lse,
                                      bool settled, cudaStream_t st) {
  if (ensure_kernel_attrs(attention_kernel<HPC>, AtPlan<HPC>::SMEM, true) != HS_OK) return HS_ERR_CUDA;
  const int n_hgrp = p->cfg.n_heads / HPC;
  return launch_pdl(attention_kernel<HPC>, dim3(n_splits, n * n_hgrp, 1), dim3(AT_THREADS, 1, 1), AtPlan<HPC>::SMEM,
                    st, n_splits, p->d, layer, d_q, d_rows, scale_log2, d_out, d_lse, settled ? 1 : 0);
}

hs_status launch_attention(hs_pool* p, int layer, int n, const uint16_t* d_q, const int32_t* d_rows, float sm_scale,
                           uint16_t* d_out, float* d_lse, bool settled, cudaStream_t st) {
  // many query tokens: one CTA per token over all its rows (hs_attention_seq.cu)
  if (attention_seq_suits(p, n)) return launch_attention_seq(p, layer, n, d_q, d_rows, sm_scale, d_out, d_lse, st);
  const int n_splits = (p->cfg.topk + ATTN_ROWS - 1) / ATTN_ROWS;
  const int H = p->cfg.n_heads;
  // fewer heads per CTA while the head groups still fit on the SMs side by side
  int hpc = H < 64 ? H : 64;
  while (hpc > 16 && (long long)n * n_splits * (H / (hpc / 2)) <= num_sms()) hpc /= 2;
  const int slice = ((512 + n_splits - 1) / n_splits + 7) & ~7;
  if (hpc == 32 && n_splits * slice > AtPlan<32>::RECV_DIMS) hpc = 16;   // receive buffer bound
  const float sl = sm_scale * LOG2E;
  if (hpc == 16) return launch_attention_hpc<16>(p, layer, n, n_splits, d_q, d_rows, sl, d_out, d_lse, settled, st);
  if (hpc == 32) return launch_attention_hpc<32>(p, layer, n, n_splits, d_q, d_rows, sl, d_out, d_lse, settled, st);
  return launch_attention_hpc<64>(p, layer, n, n_splits, d_q, d_rows, sl, d_out, d_lse, settled, st);
}

}  // namespace hs
