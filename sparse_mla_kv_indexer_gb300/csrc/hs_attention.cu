// Sparse MLA decode attention over the resolved rows, MQA form.
//
// "Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse" (vLLM blog Part 2),
// footnote 1: each query reads its 2,048 selected 656-byte FP8 rows; QK runs over
// 576 dims and PV over 512; every row serves all 64 heads (section "PCP: split
// tokens, not heads"), which is what puts sparse MLA near the compute ridge.
//
// One CTA (16 warps) per (query token, block of 128 selected rows):
//  * every thread loads ~10 of the block's 16-byte row chunks at once, gathered by
//    HMA row id (one stride for resident and hot rows), and puts each chunk in
//    place: the FP8 latent widened to bf16 by a bit shuffle that is exact up to
//    the constant factor 2^-120 (normal and subnormal e4m3 alike), the fp32 group
//    scales to a small table, the bf16 rope unchanged; the 128 x 576 bf16 tile
//    (128-byte swizzle) is the K-major A operand of QK and the MN-major A
//    operand of PV; the bf16 query is the B operand unchanged;
//  * QK on tcgen05 into five TMEM accumulators (four 128-dim latent groups and
//    the rope), so each row's per-group scales (x 2^120) are applied in fp32 when
//    the scores are read back: s = sum_g scale_g * S_g + S_rope;
//  * softmax from TMEM: each thread owns one row and 16 heads; per-head max and
//    sum over rows use a warp transpose-reduction and shared memory;
//  * PV on tcgen05 per latent group g with P_g = p * scale_g * 2^120 (bf16),
//    so the unscaled FP8 values serve as V;
//  * the CTAs of one token form a thread-block cluster: they exchange their
//    per-head (max, sum) through distributed shared memory, each CTA writes its
//    partial output, scaled by its log-sum-exp weight and rounded to fp16, to a
//    per-token merge buffer (it stays in L2), and after one cluster barrier each
//    CTA sums one slice of the 512 output dims over the splits in fp32 and
//    writes it as bf16.
// Per-group scales must stay below 256 (so scale * 2^120 fits fp32 and bf16).
#include "hs_internal.cuh"

namespace hs {

constexpr int AT_THREADS = 512;
constexpr int AT_KV_COL = ATTN_ROWS * 128;       // 16 KB: one 64-dim bf16 atom column of the tile
constexpr int AT_Q_COL = 64 * 128;               // 8 KB: one atom column of Q (<= 64 heads)
constexpr int AT_P_COL = ATTN_ROWS * 128;        // 16 KB: one P_g matrix [128 rows][64 heads] bf16
constexpr int AT_OFF_KV = 0;
constexpr int AT_OFF_Q = 9 * AT_KV_COL;          // 144 KB; after QK the region holds P_0..P_3
constexpr int AT_OFF_MISC = AT_OFF_Q + 9 * AT_Q_COL;   // 216 KB
constexpr int AT_MISC = 6144;
constexpr int AT_SMEM = AT_OFF_MISC + AT_MISC + 1024;
constexpr int AT_CHUNKS = ATTN_ROWS * ROW_CHUNKS;        // 5,248 16-byte chunks per block
constexpr int AT_CPT = (AT_CHUNKS + AT_THREADS - 1) / AT_THREADS;   // 11 per thread
constexpr float LOG2E = 1.4426950408889634f;
constexpr float TWO_POW_120 = 1.329227995784916e36f;
static_assert(4 * AT_P_COL <= 9 * AT_Q_COL, "P_0..P_3 fit in the query region");
static_assert(AT_SMEM <= 232448, "shared memory budget");

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

// After the call lanes l and l ^ 16 hold op-reduction over all 32 lanes of v[l & 15].
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      float send = hi ? v[i] : v[i + o];
      float keep = hi ? v[i + o] : v[i];
      float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float other = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return MAX ? fmaxf(v[0], other) : v[0] + other;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__global__ void __launch_bounds__(AT_THREADS, 1)
attention_kernel(Dev D, int layer, const uint16_t* __restrict__ q, const int32_t* __restrict__ row_ids,
                 float scale_log2, uint16_t* __restrict__ out, float* __restrict__ lse_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = smem + AT_OFF_KV;
  uint8_t* Qs = smem + AT_OFF_Q;
  uint8_t* Ps = smem + AT_OFF_Q;                                             // P_g after QK
  int32_t* ids = reinterpret_cast<int32_t*>(smem + AT_OFF_MISC);            // [128]
  float4* scl = reinterpret_cast<float4*>(ids + ATTN_ROWS);                  // [128] group scales
  float* red = reinterpret_cast<float*>(scl + ATTN_ROWS);                    // [4][64]
  float* mfin = red + 4 * 64;                                                // [64] this split's max (log2 units)
  float* lfin = mfin + 64;                                                   // [64] this split's sum
  float* wmine = lfin + 64;                                                  // [64] weight of this split
  float* gstat = wmine + 64;                                                 // [64] lse
  uint64_t* bar = reinterpret_cast<uint64_t*>(gstat + 64);                   // [1] MMA completion
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  int32_t* s_flag = reinterpret_cast<int32_t*>(tslot + 1);

  const uint32_t split = cluster_rank();
  const uint32_t n_splits = cluster_size();
  const int tok = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = D.n_heads, K = D.topk;
  const uint8_t* kv = D.kv[layer];
  const long long max_row = (long long)D.num_pages * PAGE;

  if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
    *s_flag = 0;
  }
  griddep_wait();
  griddep_launch();
  if (tid < ATTN_ROWS) {
    const int k = (int)split * ATTN_ROWS + tid;
    int id = k < K ? row_ids[(size_t)tok * K + k] : -1;
    if (id >= max_row) { set_status(D.status, HS_ERR_BAD_ID); id = -1; }
    ids[tid] = id;
  }
  // ---- Q: [H, 576] bf16, 72 chunks of 8 per head, loads in flight ----
  const uint16_t* qt = q + (size_t)tok * H * QK;
  constexpr int QPT = 64 * 72 / AT_THREADS;   // 9 chunks per thread at 64 heads
  uint4 qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int c = tid + k * AT_THREADS;
    qv[k] = c < H * 72 ? __ldg(reinterpret_cast<const uint4*>(qt) + c) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();   // ids ready
  // ---- all row chunks in flight at once: chunk c = row * 41 + part ----
  uint4 rc[AT_CPT];
#pragma unroll
  for (int k = 0; k < AT_CPT; ++k) {
    const int c = tid + k * AT_THREADS;
    rc[k] = make_uint4(0, 0, 0, 0);
    if (c < AT_CHUNKS) {
      const int r = c / ROW_CHUNKS, part = c - r * ROW_CHUNKS;
      const int id = ids[r];
      if (id >= 0) rc[k] = __ldg(reinterpret_cast<const uint4*>(kv + (size_t)id * ROW) + part);
    }
  }
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int c = tid + k * AT_THREADS;
    if (c < H * 72) {
      const int h = c / 72, ch = c - h * 72;
      *reinterpret_cast<uint4*>(Qs + (ch >> 3) * AT_Q_COL + sw128_chunk(h, ch & 7)) = qv[k];
    }
  }
#pragma unroll
  for (int k = 0; k < AT_CPT; ++k) {
    const int c = tid + k * AT_THREADS;
    if (c < AT_CHUNKS) {
      const int r = c / ROW_CHUNKS, part = c - r * ROW_CHUNKS;
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
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // ---- S_g^T = KV_g . Q_g^T (g = 0..3 latent groups, 4 = rope): M = 128 rows, N = H ----
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, H, false, false, true);
    const uint32_t a0 = smem_u32(KV), b0 = smem_u32(Qs);
#pragma unroll 4
    for (int kk = 0; kk < 36; ++kk) {
      const int g = kk >> 3;          // 8 k-steps of 16 dims per 128-dim group; rope is g = 4
      const uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * AT_KV_COL + (kk & 3) * 32, 16, 1024);
      const uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * AT_Q_COL + (kk & 3) * 32, 16, 1024);
      umma_f16(tmem + g * 64, ad, bd, idesc, (kk & 7) != 0);
    }
    umma_commit(smem_u32(bar));
  }
  if (!mbar_wait(smem_u32(bar), 0, D.status)) *s_flag = 1;
  tc_fence_after();

  // ---- softmax over the 128 rows, per head: warp (row quadrant, head quarter) ----
  const int quad = warp & 3, hq = warp >> 2;
  const int row = quad * 32 + lane;
  const bool valid = ids[row] >= 0;
  const bool active = hq * 16 < H;          // warp-uniform
  const float4 sc4 = scl[row];
  const float sg[4] = {sc4.x * TWO_POW_120, sc4.y * TWO_POW_120, sc4.z * TWO_POW_120, sc4.w * TWO_POW_120};
  float z[16];
  if (active) {
    const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(hq * 16);
    uint32_t r[16];
    tmem_ld16(ta + 256, r);         // rope part
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = __uint_as_float(r[i]);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      tmem_ld16(ta + g * 64, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = fmaf(__uint_as_float(r[i]), sg[g], z[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = valid ? z[i] * scale_log2 : -INFINITY;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = z[i];
    const float m = warp_transpose_reduce16<true>(t);
    if (lane < 16) red[quad * 64 + hq * 16 + lane] = m;
  }
  __syncthreads();
  if (tid < H) mfin[tid] = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
  __syncthreads();
  if (active) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float m = mfin[hq * 16 + i];
      const float p = (m == -INFINITY || z[i] == -INFINITY) ? 0.f : exp2f(z[i] - m);
      z[i] = p;
      t[i] = p;
    }
    const float l = warp_transpose_reduce16<false>(t);
    if (lane < 16) red[quad * 64 + hq * 16 + lane] = l;
    // P_g^T[row][head] = p * scale_g * 2^120 (bf16), the MN-major B operand of group g
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint8_t* pg = Ps + g * AT_P_COL;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float* zz = z + 8 * c;
        *reinterpret_cast<uint4*>(pg + sw128_chunk(row, hq * 2 + c)) =
            make_uint4(pack_bf16x2(zz[0] * sg[g], zz[1] * sg[g]), pack_bf16x2(zz[2] * sg[g], zz[3] * sg[g]),
                       pack_bf16x2(zz[4] * sg[g], zz[5] * sg[g]), pack_bf16x2(zz[6] * sg[g], zz[7] * sg[g]));
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();   // every S read: the accumulators may be overwritten by PV
  if (tid < H) lfin[tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
  tc_fence_after();

  // ---- O_g^T = V_g^T . P_g^T : M = 128 latent dims, N = H, K = 128 rows ----
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, H, true, true, true);
    const uint32_t kv0 = smem_u32(KV), p0 = smem_u32(Ps);
    for (int g = 0; g < 4; ++g) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = smem_desc_sw128(kv0 + (2 * g) * AT_KV_COL + kk * 2048, AT_KV_COL, 1024);
        const uint64_t bd = smem_desc_sw128(p0 + g * AT_P_COL + kk * 2048, AT_P_COL, 1024);
        umma_f16(tmem + g * 64, ad, bd, idesc, kk > 0);
      }
    }
    umma_commit(smem_u32(bar));
  }
  if (!mbar_wait(smem_u32(bar), 1, D.status)) *s_flag = 1;
  tc_fence_after();
  // every CTA's (max, sum) is published
  cluster_sync();
  // ---- cluster-wide log-sum-exp weight of this split, per head ----
  if (tid < H) {
    float ms[MAX_SPLITS], ls[MAX_SPLITS];
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) {          // all remote loads in flight at once
      ms[s] = s < (int)n_splits ? __uint_as_float(ld_cluster_u32(mapa(smem_u32(mfin + tid), s))) : -INFINITY;
      ls[s] = s < (int)n_splits ? __uint_as_float(ld_cluster_u32(mapa(smem_u32(lfin + tid), s))) : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s) M = fmaxf(M, ms[s]);
    float L = 0.f;
#pragma unroll
    for (int s = 0; s < MAX_SPLITS; ++s)
      if (ms[s] != -INFINITY) L += exp2f(ms[s] - M) * ls[s];
    const float mine = mfin[tid];
    wmine[tid] = (L > 0.f && mine != -INFINITY) ? exp2f(mine - M) / L : 0.f;
    gstat[tid] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  __syncthreads();

  // ---- weighted partial O (fp16) to the token's merge buffer in global memory ----
  // layout [split][dim][head] (fp16); the cluster barrier below orders these
  // writes before the other CTAs of the cluster read them (cluster scope)
  __half* part = D.o_part + (size_t)tok * MAX_SPLITS * 512 * 64;
  if (active) {
    float wv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = wmine[hq * 16 + i];
    for (int g = 0; g < 4; ++g) {
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * 64 + hq * 16);
      const int dim = g * 128 + quad * 32 + lane;
      uint32_t r[16];
      tmem_ld16(ta, r);
      tmem_wait_ld();
      uint32_t hv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        __half2 h2 = __floats2half2_rn(__uint_as_float(r[2 * i]) * wv[2 * i],
                                       __uint_as_float(r[2 * i + 1]) * wv[2 * i + 1]);
        hv[i] = *reinterpret_cast<uint32_t*>(&h2);
      }
      uint4* dst = reinterpret_cast<uint4*>(part + ((size_t)split * 512 + dim) * 64 + hq * 16);
      dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
    }
  }
  tc_fence_before();
  cluster_sync();   // every partial output written
  // ---- this CTA sums one slice of the 512 dims over the splits and writes bf16 ----
  {
    const int slice = ((512 / (int)n_splits) + 3) & ~3;
    const int d_lo = min(512, (int)split * slice), d_hi = min(512, d_lo + slice);
    const int nd = d_hi - d_lo;
    for (int e = tid; e < nd * (H / 8); e += AT_THREADS) {
      const int dd = e / (H / 8), h8 = e - dd * (H / 8);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint4 v[MAX_SPLITS];
#pragma unroll
      for (int s = 0; s < MAX_SPLITS; ++s)   // coherent loads: written during this kernel
        v[s] = s < (int)n_splits ? ld_cg_v4(part + ((size_t)s * 512 + d_lo + dd) * 64 + h8 * 8)
                                 : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int s = 0; s < MAX_SPLITS; ++s) {
        const uint32_t w[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
          acc[2 * k] += f.x;
          acc[2 * k + 1] += f.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        out[((size_t)tok * H + h8 * 8 + j) * 512 + d_lo + dd] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j]));
    }
    if (split == 0 && lse_out && tid < H) lse_out[(size_t)tok * H + tid] = gstat[tid];
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

hs_status launch_attention(hs_pool* p, int layer, int n, const uint16_t* d_q, const int32_t* d_rows, float sm_scale,
                           uint16_t* d_out, float* d_lse, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return HS_ERR_CUDA;
    attr = true;
  }
  const int n_splits = (p->cfg.topk + ATTN_ROWS - 1) / ATTN_ROWS;
  return launch_pdl(attention_kernel, dim3(n_splits, n, 1), dim3(AT_THREADS, 1, 1), AT_SMEM, st, n_splits, p->d, layer,
                    d_q, d_rows, sm_scale * LOG2E, d_out, d_lse);
}

}  // namespace hs
