// Sparse MLA decode for batches of many query tokens (MTP verification batches,
// many requests): one CTA per query token walks the token's selected rows in
// blocks of 128, with the next block's rows in flight while the current block
// is on the tensor cores.
//
// "Serving GLM-5.3 with PCP, DCP and Hybrid HiSparse" (vLLM blog Part 2),
// footnote 1 and section "PCP: split tokens, not heads": every selected 656-byte
// FP8 row serves all 64 heads of a query (MQA form), QK over 576 dims, PV over
// 512. With 64 heads and several query tokens per request the work sits near the
// bf16 ridge, so the tensor cores stay busy only if the row gather is hidden
// behind them; the split-row kernel (hs_attention.cu) runs one 128-row block per
// CTA and leaves the gather and the MMAs of a CTA back to back.
//
// Roles (512 threads, one CTA per SM, persistent over tokens):
//   warps 0-3   softmax and output: thread t owns row t of the score tile (TMEM
//               lane t) and, in the output, latent dim t of each 128-dim group
//   warp 4      TMEM allocation and the tcgen05.mma issue
//   warps 5-15  gather: the 128 rows of a block, by HMA row id, 16 bytes per load,
//               into registers one block ahead; then the fp16 operand tile
// Per block b of 128 rows:
//   gather   wait until PV(b-1) has read the tile; write the tile (pieces dealt so
//            that stores of one shared-memory cycle hit distinct banks): latent values
//            e4m3 x group scale rounded once to fp16, rope bf16 -> fp16 (exact);
//            then issue the loads of block b+1
//   MMA      S = K_b . Q^T (M = 128 rows, N = 64 heads, K = 576) into TMEM
//   softmax  z = S * sm_scale * log2(e); per-head running maximum with a lazy
//            rescale (the reference maximum moves only when a block's maximum
//            exceeds it by more than 2^8, and then O and l are rescaled in place);
//            P = 2^(z - m) in fp16 into the tile's rope columns, which QK(b) no
//            longer needs
//   MMA      O^T += V_b^T . P^T per 128-dim group (M = 128 dims, N = 64 heads,
//            K = 128 rows), O in TMEM for the whole token; and l += 1 . P^T, the
//            running sum of P per head, with an all-ones A operand held in TMEM
//            (every TMEM lane of l then holds the sums of all heads)
// After the last block: out = O / l in bf16, lse = m + log(l).
//
// Precision: the scale of each 128-value group is folded into the fp16 operand
// (the exact e4m3 value times the scale rounded to fp16, relative error within 2^-10),
// so one accumulator holds the whole score; P is
// fp16; accumulation is fp32. fp16 bounds the inputs: |group scale| < 146 (so
// 448 x scale < 65504), and the query and rope values below 65504 in magnitude;
// values outside set HS_ERR_RANGE. Every wait is bounded (HS_ERR_TIMEOUT).
#include <cuda_fp8.h>

#include "hs_internal.cuh"

namespace hs {

namespace {

constexpr int SQ_THREADS = 512;
constexpr int SQ_MMA_WARP = 4;
constexpr int SQ_GATHER_WARP0 = 5;
constexpr int SQ_GATHER = SQ_THREADS - SQ_GATHER_WARP0 * 32;                 // 352
constexpr int SQ_H = 64;                                                      // heads per CTA
constexpr int SQ_COL = ATTN_ROWS * 128;                                       // 16 KB atom column of the tile
constexpr int SQ_QCOL = SQ_H * 128;                                           // 8 KB atom column of Q
constexpr int SQ_OFF_Q = 9 * SQ_COL;                                          // tile: latent 0-7, rope 8
constexpr int SQ_OFF_MISC = SQ_OFF_Q + 9 * SQ_QCOL;
constexpr int SQ_CHUNKS = ATTN_ROWS * ROW_CHUNKS;                             // 5,248
constexpr int SQ_CPT = (SQ_CHUNKS + SQ_GATHER - 1) / SQ_GATHER;               // 15
constexpr int SQ_QCHUNKS = SQ_H * 72;                                         // 4,608
constexpr int SQ_QCPT = (SQ_QCHUNKS + SQ_GATHER - 1) / SQ_GATHER;             // 14
// misc region
constexpr int SQ_M_IDS = 0;                        // int32 [2][128]
constexpr int SQ_M_SCL = SQ_M_IDS + 2 * 128 * 4;   // float4 [128]: the rows' four group scales
constexpr int SQ_M_RED = SQ_M_SCL + 128 * 16;      // float [4][64] block maximum per warp
constexpr int SQ_M_MREF = SQ_M_RED + 4 * 64 * 4;   // float [64] reference maximum (log2 units)
constexpr int SQ_M_FAC = SQ_M_MREF + 64 * 4;       // float [64] rescale factor of this block
constexpr int SQ_M_VMASK = SQ_M_FAC + 64 * 4;      // uint32 [4] valid rows of the block
constexpr int SQ_M_FLAGS = SQ_M_VMASK + 16;        // int32 [4]: rescale, dead
constexpr int SQ_M_BAR = SQ_M_FLAGS + 16;          // uint64 [5]: tile_full, s_full, p_full, pv_done, fin
constexpr int SQ_M_TSLOT = SQ_M_BAR + 5 * 8;
constexpr int SQ_MISC = SQ_M_TSLOT + 16;
constexpr int SQ_SMEM = SQ_OFF_MISC + SQ_MISC + 1024;
static_assert(SQ_SMEM <= 232448, "shared memory budget");
static_assert(SQ_CPT * SQ_GATHER >= SQ_CHUNKS && SQ_QCPT * SQ_GATHER >= SQ_QCHUNKS, "chunk cover");
constexpr uint32_t SQ_TM_O = 0;     // O^T: 4 accumulators of 64 columns (128 dims x 64 heads)
constexpr uint32_t SQ_TM_S = 256;   // S: 128 rows x 64 heads
constexpr uint32_t SQ_TM_L = 320;   // l: 64 columns, the running sum of each head (same in every lane)
constexpr uint32_t SQ_TM_ONE = 384; // all-ones fp16 A operand of the l MMA (8 columns per 16 rows of K;
                                    // columns 384-511 are all filled with ones)
constexpr float SQ_LOG2E = 1.4426950408889634f;
constexpr float SQ_TWO_POW_120 = 1.329227995784916e36f;
constexpr float SQ_RESCALE_LOG2 = 8.f;   // lazy rescale threshold: p <= 2^8
constexpr float SQ_MAX_SCALE = 146.f;    // 448 x scale < 65504

__device__ __forceinline__ void bar_named(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// Named barrier over n threads that ORs `flag` across them: every thread leaves with
// the same answer, so a role whose threads saw a wait run out stops as one.
__device__ __forceinline__ bool bar_any(int id, int n, bool flag) {
  int out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}"
      : "=r"(out)
      : "r"(flag ? 1 : 0), "r"(id), "r"(n)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void mbar_arrive1(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// D[tmem] (+)= A . B (kind::f16) with the A operand read from tensor memory.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Four e4m3 bytes times a group scale, each rounded once to fp16. Each byte is first
// placed in an fp32 bit pattern (sign to bit 31, exponent and mantissa to bits
// 20-26), which is its value times 2^-120 for every finite code, normal or
// subnormal; s120 = scale x 2^120 restores the magnitude in the product.
__device__ __forceinline__ uint2 e4m3x4_scaled_f16(uint32_t w, float s120) {
  const float f0 = __uint_as_float(((w & 0x80u) << 24) | ((w & 0x7Fu) << 20));
  const float f1 = __uint_as_float(((w & 0x8000u) << 16) | ((w & 0x7F00u) << 12));
  const float f2 = __uint_as_float(((w & 0x800000u) << 8) | ((w & 0x7F0000u) << 4));
  const float f3 = __uint_as_float((w & 0x80000000u) | ((w & 0x7F000000u) >> 4));
  return make_uint2(h2_bits(__floats2half2_rn(f0 * s120, f1 * s120)), h2_bits(__floats2half2_rn(f2 * s120, f3 * s120)));
}

// Four e4m3 bytes times a group scale in fp16: the hardware conversion of each e4m3
// pair to fp16 (exact), then one fp16 multiply per pair by the scale rounded to fp16
// (two roundings, relative error within 2^-10). Used when the scale is a normal fp16
// value (>= 2^-14), else e4m3x4_scaled_f16.
__device__ __forceinline__ uint2 e4m3x4_times_f16(uint32_t w, __half2 s2) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  return make_uint2(h2_bits(__hmul2(__half2(lo), s2)), h2_bits(__hmul2(__half2(hi), s2)));
}

// Eight bf16 values -> eight fp16 (exact inside the fp16 range); *bad is set when a
// value is beyond it.
__device__ __forceinline__ uint4 bf16x8_to_f16(uint4 v, bool* bad) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t h = h2_bits(__floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u)));
    *bad |= (h & 0x7C00u) == 0x7C00u || (h & 0x7C000000u) == 0x7C000000u;
    o[i] = h;
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Reduce each of the 32 values over the 32 lanes of the warp; lane l then holds the
// reduction of value l (a transpose-reduction: each step hands half of the values to
// the partner lane).
template <bool MAX>
__device__ __forceinline__ float warp_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = hi ? v[i] : v[i + o];
      const float keep = hi ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// Role hand-offs poll (no suspend hint): the phases complete within a few hundred
// nanoseconds of each other, and a hardware sleep wakes later than polling sees them.
__device__ __forceinline__ bool sq_wait(uint32_t bar, uint32_t parity, int32_t* status, volatile int32_t* dead) {
  if (*dead) return false;
  if (!mbar_wait_spin(bar, parity, status)) {
    *dead = 1;
    return false;
  }
  return true;
}

__global__ void __launch_bounds__(SQ_THREADS, 1)
attention_seq_kernel(Dev D, int layer, int n_tok, const uint16_t* __restrict__ q, const int32_t* __restrict__ row_ids,
                     float scale_log2, uint16_t* __restrict__ out, float* __restrict__ lse_out) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tile = smem;
  uint8_t* Qs = smem + SQ_OFF_Q;
  uint8_t* Ps = tile + 8 * SQ_COL;   // P^T after QK: the rope columns
  uint8_t* misc = smem + SQ_OFF_MISC;
  int32_t* ids = reinterpret_cast<int32_t*>(misc + SQ_M_IDS);
  float4* scl = reinterpret_cast<float4*>(misc + SQ_M_SCL);
  float* red = reinterpret_cast<float*>(misc + SQ_M_RED);
  float* mref = reinterpret_cast<float*>(misc + SQ_M_MREF);
  float* fac = reinterpret_cast<float*>(misc + SQ_M_FAC);
  uint32_t* vmask = reinterpret_cast<uint32_t*>(misc + SQ_M_VMASK);
  volatile int32_t* f_rescale = reinterpret_cast<int32_t*>(misc + SQ_M_FLAGS);
  volatile int32_t* dead = f_rescale + 1;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + SQ_M_BAR);
  const uint32_t b_tile = smem_u32(bars), b_s = smem_u32(bars + 1), b_p = smem_u32(bars + 2),
                 b_pv = smem_u32(bars + 3), b_fin = smem_u32(bars + 4);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + SQ_M_TSLOT);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = D.topk, nb = K / ATTN_ROWS;
  const uint8_t* kv = D.kv[layer];
  const long long max_row = (long long)D.num_pages * PAGE;

  if (warp == SQ_MMA_WARP) tmem_alloc(smem_u32(tslot), 512);
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(smem_u32(bars + i), 1);
    fence_mbar_init();
    *f_rescale = 0;
    *dead = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  griddep_wait();
  griddep_launch();

  if (warp >= SQ_GATHER_WARP0) {
    // ---------------------------------- gather ----------------------------------
    const int gt0 = tid - SQ_GATHER_WARP0 * 32;
    const int gt = gt0;
    uint32_t it = 0;   // blocks this CTA has processed (the barrier phases)
    bool bad_range = false;
    for (int tok = blockIdx.x; tok < n_tok; tok += gridDim.x) {
      const int32_t* rid = row_ids + (size_t)tok * K;
      // Q and the ids are overwritten only after the previous token's last PV (and so
      // all its QKs) has completed
      const bool ok0 = it == 0 || sq_wait(b_pv, (it - 1) & 1, D.status, dead);
      if (bar_any(1, SQ_GATHER, !ok0)) break;
      for (int i = gt; i < 2 * ATTN_ROWS; i += SQ_GATHER) {
        int id = i < K ? __ldg(rid + i) : -1;
        if (id >= max_row) {
          set_status(D.status, HS_ERR_BAD_ID);
          id = -1;
        }
        ids[i] = id;
      }
      {
        const uint16_t* qt = q + (size_t)tok * SQ_H * QK;
        uint4 qv[SQ_QCPT];
#pragma unroll
        for (int k = 0; k < SQ_QCPT; ++k) {
          const int c = gt + k * SQ_GATHER;
          qv[k] = c < SQ_QCHUNKS ? __ldg(reinterpret_cast<const uint4*>(qt) + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < SQ_QCPT; ++k) {
          const int c = gt + k * SQ_GATHER;
          if (c < SQ_QCHUNKS) {
            const int h = c / 72, ch = c - h * 72;
            *reinterpret_cast<uint4*>(Qs + (ch >> 3) * SQ_QCOL + sw128_chunk(h, ch & 7)) = bf16x8_to_f16(qv[k], &bad_range);
          }
        }
      }
      bar_named(1, SQ_GATHER);   // ids of blocks 0 and 1
      uint4 rc[SQ_CPT];
#define SQ_ISSUE(BID)                                                                        \
  _Pragma("unroll") for (int k = 0; k < SQ_CPT; ++k) {                                       \
    const int c = gt + k * SQ_GATHER;                                                        \
    rc[k] = make_uint4(0, 0, 0, 0);                                                          \
    if (c < SQ_CHUNKS) {                                                                     \
      int r, part;                                                                           \
      row_piece(c, r, part);                                                                  \
      const int id = (BID)[r];                                                               \
      if (id >= 0 && id < max_row) rc[k] = __ldg(reinterpret_cast<const uint4*>(kv + (size_t)id * ROW) + part); \
    }                                                                                        \
  }
      SQ_ISSUE(ids)
      bool failed = false;
      for (int b = 0; b < nb; ++b, ++it) {
        int gt;   // opaque copy of the thread's index: the per-chunk rows and offsets are
                  // recomputed each block instead of being kept in registers for the launch
        asm volatile("mov.u32 %0, %1;" : "=r"(gt) : "r"(gt0));
        const bool okb = b == 0 || sq_wait(b_pv, (it - 1) & 1, D.status, dead);   // PV(b-1) has read the tile
        asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's id copies (visible after the barrier)
        const int32_t* bid = ids + (b & 1) * ATTN_ROWS;
        // phase A: the rows' group scales (x 2^120) and the valid-row mask
#pragma unroll
        for (int k = 0; k < SQ_CPT; ++k) {
          const int c = gt + k * SQ_GATHER;
          if (c < SQ_CHUNKS) {
            int r, part;
            row_piece(c, r, part);
            if (part == 32) {
              const float4 s = make_float4(__uint_as_float(rc[k].x), __uint_as_float(rc[k].y),
                                           __uint_as_float(rc[k].z), __uint_as_float(rc[k].w));
              bad_range |= !(fabsf(s.x) < SQ_MAX_SCALE && fabsf(s.y) < SQ_MAX_SCALE && fabsf(s.z) < SQ_MAX_SCALE &&
                             fabsf(s.w) < SQ_MAX_SCALE);
              scl[r] = s;
            }
          }
        }
        if (gt < ATTN_ROWS) {
          const int id = bid[gt];
          if (id >= max_row) set_status(D.status, HS_ERR_BAD_ID);
          const unsigned m = __ballot_sync(0xffffffffu, id >= 0 && id < max_row);
          if (lane == 0 && okb) vmask[gt >> 5] = m;
        }
        if (bar_any(1, SQ_GATHER, !okb)) {
          failed = true;
          break;
        }
        // phase B: the fp16 operand tile
#pragma unroll
        for (int k = 0; k < SQ_CPT; ++k) {
          const int c = gt + k * SQ_GATHER;
          if (c < SQ_CHUNKS) {
            int r, part;
            row_piece(c, r, part);
            const uint4 v = rc[k];
            if (part < 32) {   // latent dims 16 part .. 16 part + 15, group part / 8
              const float4 s4 = scl[r];
              const int g = part >> 3;
              const float s = g == 0 ? s4.x : g == 1 ? s4.y : g == 2 ? s4.z : s4.w;
              uint2 a, bq, cq, d;
              if (fabsf(s) >= 6.103515625e-05f) {   // 2^-14: a normal fp16 scale
                const __half2 s2 = __float2half2_rn(s);
                a = e4m3x4_times_f16(v.x, s2), bq = e4m3x4_times_f16(v.y, s2);
                cq = e4m3x4_times_f16(v.z, s2), d = e4m3x4_times_f16(v.w, s2);
              } else {
                const float s120 = s * SQ_TWO_POW_120;
                a = e4m3x4_scaled_f16(v.x, s120), bq = e4m3x4_scaled_f16(v.y, s120);
                cq = e4m3x4_scaled_f16(v.z, s120), d = e4m3x4_scaled_f16(v.w, s120);
              }
              uint8_t* col = tile + (part >> 2) * SQ_COL;
              const int chunk = (part & 3) * 2;
              *reinterpret_cast<uint4*>(col + sw128_chunk(r, chunk)) = make_uint4(a.x, a.y, bq.x, bq.y);
              *reinterpret_cast<uint4*>(col + sw128_chunk(r, chunk + 1)) = make_uint4(cq.x, cq.y, d.x, d.y);
            } else if (part > 32) {   // 8 rope values
              *reinterpret_cast<uint4*>(tile + 8 * SQ_COL + sw128_chunk(r, part - 33)) = bf16x8_to_f16(v, &bad_range);
            }
          }
        }
        fence_proxy_async();
        bar_named(1, SQ_GATHER);
        if (gt == 0) mbar_arrive1(b_tile);
        // ids of block b+2 into the buffer block b's loads came from, by asynchronous
        // copies (no thread waits for them here; they are checked when used), then
        // block b+1's loads
        if (b + 2 < nb && gt < ATTN_ROWS) {
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(ids + (b & 1) * ATTN_ROWS + gt)),
                       "l"(rid + (b + 2) * ATTN_ROWS + gt)
                       : "memory");
          asm volatile("cp.async.commit_group;" ::: "memory");
        }
        if (b + 1 < nb) {
          const int32_t* nid = ids + ((b + 1) & 1) * ATTN_ROWS;
          SQ_ISSUE(nid)
        }
      }
#undef SQ_ISSUE
      if (failed) break;
    }
    if (bad_range) set_status(D.status, HS_ERR_RANGE);
  } else if (warp == SQ_MMA_WARP) {
    // ---------------------------------- MMA issue ----------------------------------
    if (lane == 0) {
      uint32_t it = 0;
      const uint32_t idesc_qk = idesc_f16(128, SQ_H, false, false, false);
      const uint32_t idesc_pv = idesc_f16(128, SQ_H, true, true, false);
      const uint32_t idesc_l = idesc_f16(128, SQ_H, false, true, false);
      const uint32_t t0 = smem_u32(tile), q0 = smem_u32(Qs), p0 = smem_u32(Ps);
      bool failed = false;
      for (int tok = blockIdx.x; tok < n_tok && !failed; tok += gridDim.x) {
        for (int b = 0; b < nb; ++b, ++it) {
          if (!sq_wait(b_tile, it & 1, D.status, dead)) {
            failed = true;
            break;
          }
          tc_fence_after();
#pragma unroll 4
          for (int kk = 0; kk < QK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(t0 + (kk >> 2) * SQ_COL + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(q0 + (kk >> 2) * SQ_QCOL + (kk & 3) * 32, 16, 1024);
            umma_f16(tmem + SQ_TM_S, ad, bd, idesc_qk, kk > 0);
          }
          umma_commit(b_s);
          if (!sq_wait(b_p, it & 1, D.status, dead)) {
            failed = true;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int kk = 0; kk < ATTN_ROWS / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(t0 + (2 * g) * SQ_COL + kk * 2048, SQ_COL, 1024);
              const uint64_t bd = smem_desc_sw128(p0 + kk * 2048, SQ_COL, 1024);
              umma_f16(tmem + SQ_TM_O + g * 64, ad, bd, idesc_pv, (b > 0 || kk > 0) ? 1u : 0u);
            }
#pragma unroll
          for (int kk = 0; kk < ATTN_ROWS / 16; ++kk)
            umma_f16_ta(tmem + SQ_TM_L, tmem + SQ_TM_ONE + kk * 8, smem_desc_sw128(p0 + kk * 2048, SQ_COL, 1024),
                        idesc_l, (b > 0 || kk > 0) ? 1u : 0u);
          umma_commit(b_pv);
        }
      }
    }
  } else {
    // ---------------------------------- softmax and output ----------------------------------
    const int row = tid;   // 0..127: TMEM lane and tile row
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float4* mref4 = reinterpret_cast<const float4*>(mref);
    {   // the all-ones operand of the l MMA (fp16 1.0 pairs); made visible to the MMA
        // warp by the fences and the barrier before the first P hand-off
      uint32_t one[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) one[j] = 0x3C003C00u;
#pragma unroll
      for (int c = 0; c < 512 - SQ_TM_ONE; c += 32) tmem_st32(lane_base + SQ_TM_ONE + c, one);
      tmem_wait_st();
    }
    uint32_t it = 0;
    bool failed = false;
    for (int tok = blockIdx.x; tok < n_tok && !failed; tok += gridDim.x) {
      if (tid < SQ_H) mref[tid] = -INFINITY;
      bar_named(2, 128);
      for (int b = 0; b < nb; ++b, ++it) {
        const bool okb = sq_wait(b_s, it & 1, D.status, dead);
        tc_fence_after();
        const bool valid = (vmask[row >> 5] >> (row & 31)) & 1u;
        // Does any row exceed a head's reference maximum by more than the lazy bound?
        // Usually not after the first block: then the block maximum is not needed.
        bool over = false;
#pragma unroll
        for (int hh = 0; hh < 64; hh += 32) {
          uint32_t t[32];
          tmem_ld32(lane_base + SQ_TM_S + hh, t);
          tmem_wait_ld();
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 m4 = mref4[hh / 4 + h4];
            over |= __uint_as_float(t[4 * h4]) * scale_log2 > m4.x + SQ_RESCALE_LOG2;
            over |= __uint_as_float(t[4 * h4 + 1]) * scale_log2 > m4.y + SQ_RESCALE_LOG2;
            over |= __uint_as_float(t[4 * h4 + 2]) * scale_log2 > m4.z + SQ_RESCALE_LOG2;
            over |= __uint_as_float(t[4 * h4 + 3]) * scale_log2 > m4.w + SQ_RESCALE_LOG2;
          }
        }
        if (bar_any(2, 128, !okb)) {   // the role stops as one when a wait ran out
          failed = true;
          break;
        }
        const bool need_max = bar_any(2, 128, over && valid);
        if (need_max) {
          // block maximum per head, one half of the heads at a time (the reduction
          // consumes its registers; S is read again from TMEM for the exponentials)
#pragma unroll
          for (int hh = 0; hh < 64; hh += 32) {
            float t[32];
            tmem_ld32(lane_base + SQ_TM_S + hh, *reinterpret_cast<uint32_t(*)[32]>(t));
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) t[h] = valid ? t[h] * scale_log2 : -INFINITY;
            red[warp * 64 + hh + lane] = warp_reduce32<true>(t);
          }
          bar_named(2, 128);
          if (tid < SQ_H) {
            const float bm = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
            const float mo = mref[tid];
            float f = 1.f;
            if (bm > -INFINITY && (mo == -INFINITY || bm > mo + SQ_RESCALE_LOG2)) {
              if (mo != -INFINITY) {
                f = exp2f(mo - bm);
                *f_rescale = 1;
              }
              mref[tid] = bm;
            }
            fac[tid] = f;
          }
          bar_named(2, 128);
        }
        const bool rescale = need_max && *f_rescale != 0;
        float p[64];   // p = 2^(z - m)
        tmem_ld32(lane_base + SQ_TM_S, *reinterpret_cast<uint32_t(*)[32]>(p));
        tmem_ld32(lane_base + SQ_TM_S + 32, *reinterpret_cast<uint32_t(*)[32]>(p + 32));
        tmem_wait_ld();
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
          const float4 m4 = mref4[h4];
          const float m[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int h = 4 * h4 + k;
            p[h] = (!valid || m[k] == -INFINITY) ? 0.f : ex2_approx(p[h] * scale_log2 - m[k]);
          }
        }
        // P^T row: 64 heads in one 128-byte line (MN-major B operand of PV and of l)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* pp = p + 8 * c;
          *reinterpret_cast<uint4*>(Ps + sw128_chunk(row, c)) =
              make_uint4(h2_bits(__floats2half2_rn(pp[0], pp[1])), h2_bits(__floats2half2_rn(pp[2], pp[3])),
                         h2_bits(__floats2half2_rn(pp[4], pp[5])), h2_bits(__floats2half2_rn(pp[6], pp[7])));
        }
        if (rescale) {   // a block raised some head's maximum by more than 2^8: O, l *= 2^(m_old - m_new)
#pragma unroll 1
          for (int g = 0; g < 5; ++g)
#pragma unroll 1
            for (int hh = 0; hh < 64; hh += 32) {
              const uint32_t col = (g < 4 ? SQ_TM_O + g * 64 : SQ_TM_L) + hh;
              uint32_t o[32];
              tmem_ld32(lane_base + col, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * fac[hh + j]);
              tmem_st32(lane_base + col, o);
            }
          tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        bar_named(2, 128);
        if (tid == 0) {
          *f_rescale = 0;
          mbar_arrive1(b_p);
        }
      }
      if (failed) break;
      const bool okl = sq_wait(b_pv, (it - 1) & 1, D.status, dead);
      tc_fence_after();
      if (bar_any(2, 128, !okl)) break;
      // out[tok][h][128 g + t] = O_g[t][h] / l[h]; this thread's lane of l holds every head
      uint16_t* ot = out + (size_t)tok * SQ_H * 512 + warp * 32 + lane;
#pragma unroll 1
      for (int hh = 0; hh < 64; hh += 32) {
        uint32_t l[32];
        tmem_ld32(lane_base + SQ_TM_L + hh, l);
        tmem_wait_ld();
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint32_t o[32];
          tmem_ld32(lane_base + SQ_TM_O + g * 64 + hh, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float lj = __uint_as_float(l[j]);
            ot[(size_t)(hh + j) * 512 + g * 128] =
                __bfloat16_as_ushort(__float2bfloat16_rn(lj > 0.f ? __uint_as_float(o[j]) / lj : 0.f));
          }
        }
        if (lse_out && warp == (hh >> 5)) {   // warp 0 the heads 0-31, warp 1 the heads 32-63
          float lh = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) lh = j == lane ? __uint_as_float(l[j]) : lh;
          const int h = hh + lane;
          lse_out[(size_t)tok * SQ_H + h] = lh > 0.f ? (mref[h] + log2f(lh)) * 0.6931471805599453f : -INFINITY;
        }
      }
      tc_fence_before();
      bar_named(2, 128);   // every O and l read before the next token's first PV and init
    }
  }
  __syncthreads();
  if (warp == SQ_MMA_WARP && lane == 0) {   // every issued MMA has completed before TMEM is freed
    umma_commit(b_fin);
    mbar_wait(b_fin, 0, D.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == SQ_MMA_WARP) tmem_dealloc(tmem, 512);
}

}  // namespace

bool attention_seq_suits(const hs_pool* p, int n) {
  const int n_splits = p->cfg.topk / ATTN_ROWS;
  // the split-row kernel would need more than two waves of one-CTA-per-SM launches
  return p->cfg.n_heads == SQ_H && (long long)n * n_splits > 2ll * num_sms();
}

hs_status launch_attention_seq(hs_pool* p, int layer, int n, const uint16_t* d_q, const int32_t* d_rows,
                               float sm_scale, uint16_t* d_out, float* d_lse, cudaStream_t st) {
  if (ensure_kernel_attrs(attention_seq_kernel, SQ_SMEM) != HS_OK) return HS_ERR_CUDA;
  const int grid = n < num_sms() ? n : num_sms();
  return launch_pdl(attention_seq_kernel, dim3(grid), dim3(SQ_THREADS), SQ_SMEM, st, 0, p->d, layer, n, d_q, d_rows,
                    sm_scale * SQ_LOG2E, d_out, d_lse);
}

}  // namespace hs
