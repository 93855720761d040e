// Sparse MLA decode attention over the resolved rows, MQA form.
//
// "Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse" (vLLM blog Part 2),
// footnote 1: each query reads its 2,048 selected 656-byte FP8 rows; QK runs over
// 576 dims and PV over 512; every row serves all 64 heads (section "PCP: split
// tokens, not heads"), which is what puts sparse MLA near the compute ridge.
//
// One CTA per (query token, block of 128 selected rows):
//  * the rows are gathered by HMA row id (one stride for resident and hot rows),
//    the FP8 latent is decoded and scaled by its per-128 fp32 scale, the bf16 rope
//    widened, into a 128 x 576 fp16 tile in the 128-byte-swizzled layout; the
//    same tile is the K-major A operand of QK and the MN-major A operand of PV;
//  * S^T = KV . Q^T on tcgen05 (M = 128 rows, N = heads, K = 576) into tensor
//    memory; each thread owns one row and reads its scores, the per-head max and
//    sum over rows use a warp transpose-reduction and shared memory;
//  * P^T (fp16) overwrites the rope columns of the tile; O^T = V^T . P^T on
//    tcgen05 (M = 128 latent dims per group, N = heads, K = 128 rows);
//  * the CTAs of one token form a thread-block cluster: they exchange their
//    per-head (max, sum) through distributed shared memory, scale their partial
//    outputs by their log-sum-exp weights into shared memory, and each CTA sums
//    one slice of the 512 output dims over the cluster and writes it as bf16.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {

constexpr int AT_THREADS = 256;
constexpr int AT_KV_COL = ATTN_ROWS * 128;       // 16 KB: one 64-dim fp16 atom column of the tile
constexpr int AT_Q_COL = 64 * 128;               // 8 KB: one atom column of Q (<= 64 heads)
constexpr int AT_OFF_KV = 0;
constexpr int AT_OFF_Q = 9 * AT_KV_COL;          // 144 KB
constexpr int AT_OFF_MISC = AT_OFF_Q + 9 * AT_Q_COL;   // 216 KB
constexpr int AT_SMEM = AT_OFF_MISC + 4096 + 1024;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t h, float s) {
  __half2 x = *reinterpret_cast<__half2*>(&h);
  float2 f = __half22float2(x);
  __half2 y = __floats2half2_rn(f.x * s, f.y * s);
  return *reinterpret_cast<uint32_t*>(&y);
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  __half2 y = __floats2half2_rn(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
  return *reinterpret_cast<uint32_t*>(&y);
}

// After the call lane l holds op-reduction over all 32 lanes of v[l] (N = 32).
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      float send = hi ? v[i] : v[i + o];
      float keep = hi ? v[i + o] : v[i];
      float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

__global__ void __launch_bounds__(AT_THREADS, 1)
attention_kernel(Dev D, int layer, const uint16_t* __restrict__ q, const int32_t* __restrict__ row_ids,
                 float scale_log2, uint16_t* __restrict__ out, float* __restrict__ lse_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* KV = smem + AT_OFF_KV;
  uint8_t* Qs = smem + AT_OFF_Q;
  int32_t* ids = reinterpret_cast<int32_t*>(smem + AT_OFF_MISC);            // [128]
  float* red = reinterpret_cast<float*>(ids + ATTN_ROWS);                    // [4][64]
  float* mfin = red + 4 * 64;                                                // [64] this split's max (log2 units)
  float* lfin = mfin + 64;                                                   // [64] this split's sum
  float* wmine = lfin + 64;                                                  // [64] weight of this split
  float* gstat = wmine + 64;                                                 // [64] spare, [64] lse
  uint64_t* bar = reinterpret_cast<uint64_t*>(gstat + 128);                  // [1]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  int32_t* s_flag = reinterpret_cast<int32_t*>(tslot + 1);
  float* Ofull = reinterpret_cast<float*>(KV);                               // [H][512] after PV

  cg::cluster_group cluster = cg::this_cluster();
  const int split = (int)cluster.block_rank();
  const int n_splits = (int)cluster.num_blocks();
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
  for (int r = tid; r < ATTN_ROWS; r += AT_THREADS) {
    int k = split * ATTN_ROWS + r;
    int id = k < K ? row_ids[(size_t)tok * K + k] : -1;
    if (id >= max_row) { set_status(D.status, HS_ERR_BAD_ID); id = -1; }
    ids[r] = id;
  }
  // ---- Q loads in flight: [H, 576] bf16, 72 chunks of 8 per head ----
  const uint16_t* qt = q + (size_t)tok * H * QK;
  constexpr int QPT = 64 * 72 / AT_THREADS;   // 18 chunks per thread at 64 heads
  uint4 qv[QPT];
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int c = tid + k * AT_THREADS;
    qv[k] = c < H * 72 ? __ldg(reinterpret_cast<const uint4*>(qt) + c) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();   // ids ready

  // ---- gather rows: warp w takes rows 16w .. 16w+15 in two batches of 8 ----
  const int r0 = warp * 16;
  uint4 lat[8], sc[8], rp[8];
  auto load_rows = [&](int rb) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int id = ids[r0 + rb + u];
      lat[u] = make_uint4(0, 0, 0, 0);
      sc[u] = make_uint4(0, 0, 0, 0);
      rp[u] = make_uint4(0, 0, 0, 0);
      if (id >= 0) {
        const uint8_t* row = kv + (size_t)id * ROW;
        lat[u] = __ldg(reinterpret_cast<const uint4*>(row + lane * 16));
        sc[u] = __ldg(reinterpret_cast<const uint4*>(row + LATENT));
        if (lane < 8) rp[u] = __ldg(reinterpret_cast<const uint4*>(row + LATENT + 16 + lane * 16));
      }
    }
  };
  auto store_rows = [&](int rb) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int r = r0 + rb + u;
      const int g = lane >> 3;   // lane's 16 latent dims belong to scale group lane / 8
      const float s = __uint_as_float(g == 0 ? sc[u].x : g == 1 ? sc[u].y : g == 2 ? sc[u].z : sc[u].w);
      const uint32_t w[4] = {lat[u].x, lat[u].y, lat[u].z, lat[u].w};
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[2 * k] = scale_f16x2(e4m3x2_to_f16x2((uint16_t)(w[k] & 0xffff)), s);
        h[2 * k + 1] = scale_f16x2(e4m3x2_to_f16x2((uint16_t)(w[k] >> 16)), s);
      }
      uint8_t* col = KV + (lane >> 2) * AT_KV_COL;
      const int chunk = (lane & 3) * 2;
      *reinterpret_cast<uint4*>(col + sw128_chunk(r, chunk)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(col + sw128_chunk(r, chunk + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
      if (lane < 8) {
        uint4 o = make_uint4(bf16x2_to_f16x2(rp[u].x), bf16x2_to_f16x2(rp[u].y), bf16x2_to_f16x2(rp[u].z),
                             bf16x2_to_f16x2(rp[u].w));
        *reinterpret_cast<uint4*>(KV + 8 * AT_KV_COL + sw128_chunk(r, lane)) = o;
      }
    }
  };
  load_rows(0);
  // Q: bf16 -> fp16, K-major SW128, one atom column per 64 dims
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    const int c = tid + k * AT_THREADS;
    if (c < H * 72) {
      const int h = c / 72, ch = c - h * 72;
      const uint4 v = qv[k];
      uint4 o = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
      *reinterpret_cast<uint4*>(Qs + (ch >> 3) * AT_Q_COL + sw128_chunk(h, ch & 7)) = o;
    }
  }
  store_rows(0);
  load_rows(8);
  store_rows(8);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // ---- S^T = KV . Q^T : M = 128 rows, N = H, K = 576 ----
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, H, false, false);
    const uint32_t a0 = smem_u32(KV), b0 = smem_u32(Qs);
#pragma unroll 4
    for (int kk = 0; kk < 36; ++kk) {
      uint64_t ad = smem_desc_sw128(a0 + (kk >> 2) * AT_KV_COL + (kk & 3) * 32, 16, 1024);
      uint64_t bd = smem_desc_sw128(b0 + (kk >> 2) * AT_Q_COL + (kk & 3) * 32, 16, 1024);
      umma_f16(tmem, ad, bd, idesc, kk > 0);
    }
    umma_commit(smem_u32(bar));
  }
  if (!mbar_wait(smem_u32(bar), 0, D.status)) *s_flag = 1;
  tc_fence_after();

  // ---- softmax over the 128 rows, per head ----
  const int quad = warp & 3, hh = warp >> 2;
  const int row = quad * 32 + lane;
  const bool valid = ids[row] >= 0;
  const bool active = hh * 32 < H;          // warp-uniform
  const int nh = min(32, H - hh * 32);      // 16 or 32 when active
  float z[32];
  if (active) {
    const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(hh * 32);
    if (nh == 32) {
      uint32_t r[32];
      tmem_ld32(ta, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = valid ? __uint_as_float(r[i]) * scale_log2 : -INFINITY;
    } else {
      uint32_t r[16];
      tmem_ld16(ta, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = valid ? __uint_as_float(r[i]) * scale_log2 : -INFINITY;
#pragma unroll
      for (int i = 16; i < 32; ++i) z[i] = -INFINITY;
    }
    float t[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) t[i] = z[i];
    red[quad * 64 + hh * 32 + lane] = warp_transpose_reduce32<true>(t);
  }
  __syncthreads();
  if (tid < H) mfin[tid] = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
  __syncthreads();
  if (active) {
    float t[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float m = (i < nh) ? mfin[hh * 32 + i] : -INFINITY;
      const float p = (m == -INFINITY || z[i] == -INFINITY) ? 0.f : exp2f(z[i] - m);
      z[i] = p;
      t[i] = p;
    }
    red[quad * 64 + hh * 32 + lane] = warp_transpose_reduce32<false>(t);
    // P^T[row][head] as fp16 into the rope atom column (B operand, MN-major)
    uint8_t* pcol = KV + 8 * AT_KV_COL;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c * 8 < nh) {
        __half2 a = __floats2half2_rn(z[8 * c + 0], z[8 * c + 1]);
        __half2 b = __floats2half2_rn(z[8 * c + 2], z[8 * c + 3]);
        __half2 d = __floats2half2_rn(z[8 * c + 4], z[8 * c + 5]);
        __half2 e = __floats2half2_rn(z[8 * c + 6], z[8 * c + 7]);
        *reinterpret_cast<uint4*>(pcol + sw128_chunk(row, hh * 4 + c)) =
            make_uint4(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b),
                       *reinterpret_cast<uint32_t*>(&d), *reinterpret_cast<uint32_t*>(&e));
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (tid < H) lfin[tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
  tc_fence_after();

  // ---- O^T = V^T . P^T : 4 groups of M = 128 latent dims, N = H, K = 128 rows ----
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, H, true, true);
    const uint32_t kv0 = smem_u32(KV), p0 = smem_u32(KV + 8 * AT_KV_COL);
    for (int g = 0; g < 4; ++g) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint64_t ad = smem_desc_sw128(kv0 + (2 * g) * AT_KV_COL + kk * 2048, AT_KV_COL, 1024);
        uint64_t bd = smem_desc_sw128(p0 + kk * 2048, AT_KV_COL, 1024);
        umma_f16(tmem + 64 + g * 64, ad, bd, idesc, kk > 0);
      }
    }
    umma_commit(smem_u32(bar));
  }
  // (max, sum) of this split are published to the cluster while the PV product runs
  cluster.sync();
  // ---- cluster-wide log-sum-exp weight of this split, per head ----
  if (tid < H) {
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, cluster.map_shared_rank(mfin, s)[tid]);
    float L = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      const float ms = cluster.map_shared_rank(mfin, s)[tid];
      if (ms != -INFINITY) L += exp2f(ms - M) * cluster.map_shared_rank(lfin, s)[tid];
    }
    const float mine = mfin[tid];
    wmine[tid] = (L > 0.f && mine != -INFINITY) ? exp2f(mine - M) / L : 0.f;
    gstat[64 + tid] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  if (!mbar_wait(smem_u32(bar), 1, D.status)) *s_flag = 1;
  tc_fence_after();
  __syncthreads();

  // ---- weighted partial O[head][dim] (fp32) into this CTA's shared memory ----
  if (active) {
    for (int g = 0; g < 4; ++g) {
      const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(64 + g * 64 + hh * 32);
      const int dim = g * 128 + quad * 32 + lane;
      if (nh == 32) {
        uint32_t r[32];
        tmem_ld32(ta, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) Ofull[(hh * 32 + i) * 512 + dim] = __uint_as_float(r[i]) * wmine[hh * 32 + i];
      } else {
        uint32_t r[16];
        tmem_ld16(ta, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) Ofull[(hh * 32 + i) * 512 + dim] = __uint_as_float(r[i]) * wmine[hh * 32 + i];
      }
    }
  }
  tc_fence_before();
  cluster.sync();
  // ---- this CTA sums one slice of the 512 dims over the cluster and writes bf16 ----
  {
    const int slice = ((512 / n_splits) + 3) & ~3;
    const int d_lo = min(512, split * slice), d_hi = min(512, d_lo + slice);
    const int per_head = (d_hi - d_lo) / 4;          // float4s per head in the slice
    for (int e = tid; e < H * per_head; e += AT_THREADS) {
      const int h = e / per_head, d = d_lo + (e - h * per_head) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < n_splits; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(cluster.map_shared_rank(Ofull, s) + h * 512 + d);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(acc.z, acc.w);
      *reinterpret_cast<uint2*>(out + ((size_t)tok * H + h) * 512 + d) =
          make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
    if (split == 0 && lse_out && tid < H) lse_out[(size_t)tok * H + tid] = gstat[64 + tid];
  }
  cluster.sync();   // peers read this CTA's shared memory until here
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
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(n_splits, n, 1);
  lc.blockDim = dim3(AT_THREADS, 1, 1);
  lc.dynamicSmemBytes = AT_SMEM;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = n_splits;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, attention_kernel, p->d, layer, d_q, d_rows, sm_scale * LOG2E, d_out, d_lse) !=
      cudaSuccess)
    return HS_ERR_CUDA;
  return HS_OK;
}

}  // namespace hs
