// Private definitions shared by the translation units of libhisparse.so:
// pool state, geometry constants and the sm_103a PTX wrappers (mbarrier,
// bulk copies, tcgen05 tensor-core and tensor-memory instructions).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "hisparse.h"

namespace hs {

constexpr int PAGE = 64;           // tokens per page
constexpr int ROW = 656;           // bytes per KV row
constexpr int ROW_CHUNKS = 41;     // 16-byte chunks per row
constexpr int LATENT = 512;        // FP8 latent dims
constexpr int ROPE = 64;           // bf16 rope dims
constexpr int QK = 576;            // QK dims
constexpr int IDX_DIM = 128;       // index key dims
constexpr int IDX_PAGE_BYTES = PAGE * IDX_DIM;
constexpr int ATTN_ROWS = 128;     // selected rows per attention CTA (MMA M)
constexpr int MAX_SPLITS = 16;     // 2048 / 128
constexpr uint64_t WAIT_NS = 1000000000ull;   // bounded device waits: 1 s

// Device-side view of a pool (passed by value to kernels).
struct Dev {
  // geometry
  int32_t n_idx_heads, n_heads, topk, n_layers, lpi, n_groups;
  int32_t num_pages, num_idx_pages, max_requests, max_ctx, max_pages;
  int32_t max_q, hot_rows, hot_pages_max, max_tokens;
  int32_t idx_fmt, idx_page_bytes;   // HS_IDX_INT8 / HS_IDX_FP8 and the key-cache page size
  int64_t host_pages;
  // residency metadata
  int32_t* bt;          // [max_requests, max_pages] pool page or -1
  int32_t* idx_bt;      // [max_requests, max_pages] index-cache page
  int64_t* host_pg;     // [max_requests, max_pages] host page or -1
  int32_t* hot_pages;   // [max_requests, n_groups, hot_pages_max]
  int32_t* n_hot;       // [max_requests, n_groups] leased pages
  int32_t* slot_token;  // [max_requests, n_groups, hot_rows]
  int32_t* slot_stamp;  // [max_requests, n_groups, hot_rows]
  int32_t* tok2slot;    // [max_requests, n_groups, max_ctx]
  // caller-owned data
  uint8_t** kv;         // [n_layers] device pointers
  int8_t** idx;         // [n_groups] device pointers
  uint8_t* host;        // device alias of the pinned host pool
  // status and counters
  int32_t* status;
  unsigned long long* counters;   // resident, hits, misses, h2d, d2h
  // scratch
  int64_t* scores;      // [max_tokens, max_ctx]
  __half* o_part;       // [max_tokens, MAX_SPLITS, 512, 64] fp16 partial attention outputs
  float2* o_stats;      // [max_tokens, MAX_SPLITS, 64] per split and head: (max in log2 units, sum)
  uint8_t* sel_ws;      // [sel_ws_tokens] SelWs: wide top-K selection scratch, zero between launches
  int32_t sel_ws_tokens;
  uint8_t* bsel;        // [bsel_tokens] BselTok: chunked selection scratch (many query tokens)
  int32_t bsel_tokens;
};

enum Counter { C_RESIDENT = 0, C_HITS = 1, C_MISSES = 2, C_H2D = 3, C_D2H = 4, C_N = 8 };

}  // namespace hs

struct hs_pool {
  hs_pool_config cfg;
  hs::Dev d;
  int device;
  std::vector<int32_t> n_hot_host;   // leased pages per (req, group), mirrored on the host
  std::vector<void*> allocations;
  // HS_IDX_FP8, three per indexer layer: one page's 64 key rows (2-D, 128-byte
  // swizzled), two adjacent pages' key rows (3-D: the scale rows between them are
  // skipped), two adjacent pages' scales (2-D, 256 bytes per page)
  std::vector<CUtensorMap> idx_tmaps;
  // The last hot-path launch of this pool was hs_sparse_mla_decode over settled_rows
  // on settled_stream (null: it was something else). A decode that follows it with
  // the same rows on the same stream may read them before that kernel completes.
  const void* settled_rows = nullptr;
  void* settled_stream = nullptr;
  int32_t select_mode = HS_SELECT_AUTO;   // hs_set_select_mode
};

namespace hs {

// ---- error helpers ---------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t* st, int code) {
  atomicCAS(st, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// One bounded test of a phase: the warp may sleep in hardware until the phase
// completes or the suspend hint (ns) expires, instead of spinning in issue slots.
constexpr uint32_t MBAR_SUSPEND_NS = 20000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(MBAR_SUSPEND_NS)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of a barrier, giving up after WAIT_NS and recording
// HS_ERR_TIMEOUT. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {   // each test may sleep up to MBAR_SUSPEND_NS
      uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > WAIT_NS) {
        set_status(status, HS_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// The same wait polling without the suspend hint: for a short pipeline whose
// phases complete within a few hundred ns, a hardware sleep wakes up later than
// polling notices the phase.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, int32_t* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 255u) == 0) {
      uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > WAIT_NS) {
        set_status(status, HS_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---- bulk copies (TMA unit, untiled) ------------------------------------------
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// 2-D tiled tensor load (TMA) of the box at (x, y) into shared memory, completing
// bytes on `bar`; the tensor map is a __grid_constant__ kernel parameter.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// 3-D tiled tensor load (TMA) of the box at (x, y, z).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 ---------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] x B[smem desc], kind::f16, issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A . B with e4m3 operands (kind::f8f6f4; K = 32 per instruction).
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Each thread of the warp reads 32 consecutive fp32 columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
// N consecutive fp32 columns (N = 4, 8, 16, 32 or 64) of the thread's own lane,
// issued without waiting; the caller waits once with tmem_wait_ld().
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  static_assert(N == 4 || N == 8 || N == 16 || N == 32 || N == 64, "column count");
  if constexpr (N == 4) {
    tmem_ld4(taddr, r);
  } else if constexpr (N == 8) {
    tmem_ld8(taddr, r);
  } else if constexpr (N == 16) {
    tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
  } else {
#pragma unroll
    for (int j = 0; j < N / 32; ++j) tmem_ld32(taddr + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * j));
  }
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//  K-major operand: rows of 128 B (64 16-bit elements), 8-row groups `sbo` apart.
//  MN-major operand: 128-B lines of 64 MN elements, 8 K-lines per group `sbo`
//  apart, 64-element MN blocks `lbo` apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;          // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;          // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16 with fp16 (or bf16) A and B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major,
                                                 bool bf16 = false) {
  return (1u << 4)                                   // D = f32
         | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10)   // A, B = f16 or bf16
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// kind::f8f6f4 with e4m3 A and B (format code 0 in both operand fields) and f32 D:
// the same bits as f16 x f16 -> f32; only the MMA's kind differs.
__host__ __device__ constexpr uint32_t idesc_f8_e4m3(int M, int N) { return idesc_f16(M, N, false, false, false); }

// ---- distributed shared memory (thread-block clusters) ---------------------------
// Cluster-wide barrier with release/acquire ordering of shared-memory accesses.
// Split-phase cluster barrier: every thread of every CTA of the cluster arrives,
// then waits. A relaxed arrival orders nothing; it only says "this CTA has started",
// which must hold for every CTA before any of them touches another's shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Asynchronous stores into another CTA's shared memory; each completes `bytes` of
// the transaction count of that CTA's mbarrier `rbar` (both cluster addresses).
__device__ __forceinline__ void st_async_v2f(uint32_t raddr, float x, float y, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
               "f"(x), "f"(y), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   raddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_cluster_v2f(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ float2 ld_cg_f2(const void* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}
// 16-byte global load that bypasses the non-coherent path (data written by this kernel).
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

// Byte offset of 16-bit element (row, col) inside a [rows x 64] SW128 block
// (row-major 128-B lines, 16-B chunks XOR-swizzled by row % 8).
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) & 7) << 4) + ((col & 7) << 1));
}
// Byte offset of the 16-B chunk `chunk` (0..7) of line `row`.
__host__ __device__ __forceinline__ uint32_t sw128_chunk(int row, int chunk) {
  return (uint32_t)(row * 128 + (((chunk ^ (row & 7)) & 7) << 4));
}

// The 5,248 16-byte pieces of a 128-row attention block (128 rows x 41 parts), in the
// order the gathering threads of a CTA take them (slot c goes to thread c % threads,
// a multiple of 32): the row and the 16-byte part of the 656-byte row it holds. Every group of 8 consecutive slots (8 threads that store in
// one shared-memory cycle) covers 4 parts of two rows whose swizzled 16-byte slots
// differ, so the group's 16-byte stores of the fp16 tile fall on 8 different bank
// groups, and a warp's loads cover two runs of 256 contiguous bytes.
//   slots [0, 4096)     latent parts 0-31: rows 2P, 2P + 1 (P = c / 64), parts 4j .. 4j + 3
//   slots [4096, 5120)  rope parts 33-40: rows 8G + q and 8G + q + 4, four parts each
//   slots [5120, 5248)  part 32 (the four group scales) of row c - 5120
__host__ __device__ __forceinline__ void row_piece(int c, int& r, int& part) {
  if (c < 4096) {
    const int u = c >> 3, t = c & 7;
    r = 2 * (u >> 3) + (t >> 2);
    part = 4 * (u & 7) + (t & 3);
  } else if (c < 5120) {
    const int u = (c - 4096) >> 3, t = c & 7;
    r = 8 * (u >> 3) + ((u >> 1) & 3) + 4 * (t >> 2);
    part = 33 + 4 * (u & 1) + (t & 3);
  } else {
    r = c - 5120;
    part = 32;
  }
}

// ---- programmatic dependent launch -------------------------------------------------
// A hot-path kernel may start while its predecessor in the stream finishes; it
// runs its address-independent prologue, then waits for the predecessor's
// completion (and memory) before touching global data, then lets its own
// successor start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline hs_status launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    dim3 cluster, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute at[2];
  int na = 0;
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster.x * cluster.y * cluster.z > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = cluster.x;
    at[na].val.clusterDim.y = cluster.y;
    at[na].val.clusterDim.z = cluster.z;
    ++na;
  }
  lc.attrs = at;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
// clusters of `cluster_x` CTAs along x (0: no cluster)
template <typename... KArgs, typename... Args>
inline hs_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            int cluster_x, Args... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, st, dim3(cluster_x > 0 ? cluster_x : 1, 1, 1), args...);
}

// ---- kernel attributes, set once per (kernel, device) -------------------------------
// Raises `kernel`'s dynamic shared-memory limit to at least `smem` bytes (and allows
// cluster sizes above 8 when asked) on the current device, once per device: the
// attributes are per device, and a process may drive pools on several GPUs.
hs_status ensure_kernel_attrs(const void* kernel, int smem, bool nonportable_cluster);
template <typename... KArgs>
inline hs_status ensure_kernel_attrs(void (*kernel)(KArgs...), int smem, bool nonportable_cluster = false) {
  return ensure_kernel_attrs(reinterpret_cast<const void*>(kernel), smem, nonportable_cluster);
}

// ---- host-side launch helpers (defined in hs_pool.cu) ----------------------------
// d_hist0: nullable; the selection's level-0 histogram sums, which the scoring
// kernel fills when the selection runs wide for one query token (select_hist0)
hs_status launch_indexer(hs_pool* p, int il, int n, const int32_t* d_req, const int32_t* d_limit,
                         const int8_t* d_q, const int8_t* d_w, int64_t* d_scores, uint32_t* d_hist0,
                         cudaStream_t st);
// CTAs per query token of the wide selection of n tokens (0: the cluster selection)
int select_wide_groups(hs_pool* p, int n, bool wide_ok);
// The level-0 histogram sums the scoring kernel fills for a wide one-token selection, else null.
uint32_t* select_hist0(hs_pool* p, int n, bool wide_ok);
// fp_keys: the scores are order-preserving keys of fp32 scores (FP8 indexer);
// wide_ok: the pool's selection scratch may be used (few tokens: the wide kernel);
// hist0_done: the scoring kernel filled select_hist0()
hs_status launch_select(hs_pool* p, int n, const int64_t* scores, int ld, const int32_t* d_limit,
                        int32_t* d_topk, cudaStream_t st, bool fp_keys = false, bool wide_ok = true,
                        bool hist0_done = false);
hs_status launch_resolve(hs_pool* p, int group, int step, int n, const int32_t* d_req,
                         const int32_t* d_topk, int32_t* d_row_ids, hs_plan_entry* d_plan,
                         cudaStream_t st);
hs_status launch_indexer_fp8(hs_pool* p, int il, int n, const int32_t* d_req, const int32_t* d_limit,
                             const uint8_t* d_q, const float* d_w, int64_t* d_keys, float* d_scores,
                             uint32_t* d_hist0, cudaStream_t st);
hs_status launch_replay(hs_pool* p, int group, int n, const int32_t* d_req, const int32_t* d_topk,
                        int32_t* d_row_ids, cudaStream_t st);
// settled: d_rows and the rows it names were written before the previous kernel of
// the stream, which is a decode of the same rows (see hs_pool::settled_rows)
hs_status launch_attention(hs_pool* p, int layer, int n, const uint16_t* d_q, const int32_t* d_rows,
                           float sm_scale, uint16_t* d_out, float* d_lse, bool settled, cudaStream_t st);
// the one-CTA-per-token attention for many query tokens (64 heads)
bool attention_seq_suits(const hs_pool* p, int n);
hs_status launch_attention_seq(hs_pool* p, int layer, int n, const uint16_t* d_q, const int32_t* d_rows,
                               float sm_scale, uint16_t* d_out, float* d_lse, cudaStream_t st);
int num_sms();

}  // namespace hs
