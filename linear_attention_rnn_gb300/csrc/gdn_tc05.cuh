// gdn_tc05.cuh -- 5th-generation tensor-core (tcgen05) helpers for sm_103a.
//
// Operands live in shared memory in the K-major, 128-byte-swizzled canonical
// layout: a [rows x 128] bf16 tile is stored as two 64-column halves, each
// rows x 128 B, and within a half the 16-byte chunk j of row r sits at chunk
// position j ^ (r % 8).  A matrix descriptor points at one half (plus 32 B per
// 16-element k step); the stride between 8-row groups is 1024 B.  The
// accumulator lives in tensor memory (TMEM): for M = 128, row m of D is TMEM
// lane m and column n is TMEM column base + n (fp32).
#pragma once
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {
namespace tc {

// byte offset of element (r, c) in a [rows x 128] bf16 K-major SW128 tile
__device__ __forceinline__ uint32_t sw128(int r, int c, int rows) {
  const int half = c >> 6, cc = c & 63;
  return (uint32_t)(half * rows * 128 + r * 128 + ((((cc >> 3) ^ (r & 7))) << 4) + ((cc & 7) << 1));
}
// byte offset of the 16-byte chunk j (columns 8j..8j+7) of row r
__device__ __forceinline__ uint32_t sw128_chunk(int r, int j, int rows) {
  const int half = j >> 3;
  return (uint32_t)(half * rows * 128 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// shared-memory matrix descriptor: start address, LBO (unused for swizzled
// K-major), SBO = 1024 B, descriptor version 1, 128-byte swizzle
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// instruction descriptor: kind::f16, A = B = bf16 (K-major), D = fp32
__device__ __forceinline__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}

// D[128 x N] (+)= A[128 x 16 NK] * B[N x 16 NK]^T, both K-major SW128 tiles
// (A with 128 rows, B with N rows; NK = 8: K = 128 over both 64-column halves,
// NK = 4: K = 64, the first half only); issued by one thread.
template <int NK = 8>
__device__ __forceinline__ void gemm_k128(uint32_t tmem_d, uint32_t a_smem, uint32_t b_smem,
                                          int N, bool accumulate_first) {
  const uint32_t idesc = (N == 128) ? idesc_bf16(128, 128) : idesc_bf16(128, N);
  // the descriptors are linear in the address (bits 0-13 hold address / 16, and
  // every operand lies inside the CTA's shared memory, below 256 KiB): each
  // step adds its constant offset to the base descriptors
  const uint64_t da0 = desc_sw128(a_smem), db0 = desc_sw128(b_smem);
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    const uint32_t koff = (uint32_t)(k & 3) * 32u;
    const uint64_t da = da0 + (((uint32_t)(k >> 2) * 128u * 128u + koff) >> 4);
    const uint64_t db = db0 + (((uint32_t)(k >> 2) * (uint32_t)N * 128u + koff) >> 4);
    mma(tmem_d, da, db, idesc, (k > 0 || accumulate_first) ? 1u : 0u);
  }
}

__device__ __forceinline__ void commit(uint64_t* mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(mbar))
               : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// make generic-proxy shared-memory writes visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32(w%4)..+31)
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- mbarriers --------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Every wait of this library's kernels gives up after this many SM cycles
// (about one second at the GB300's 2.07 GHz, longer at lower clocks).  A wait
// is for a TMA copy, an MMA or a handshake inside one CTA, normally
// microseconds.
constexpr long long WAIT_LIMIT_CYCLES = 2000000000LL;
// Waits for the phase with the given parity to complete; gives up after
// limit_cycles SM cycles and returns false (the caller records an error).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          long long limit_cycles = WAIT_LIMIT_CYCLES) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (clock64() - t0 > limit_cycles) return false;
  }
}

// try_wait with a suspend-time hint (ns): the thread sleeps until the phase
// completes or the hint runs out, instead of spinning.  Spinning waiters take
// issue slots from the threads that issue the products and copies.  Measured
// per kernel: it pays for every wait of the walks and the preparation and for
// the gradient kernel's many-thread waits; the gradient kernel's issuing
// thread, which waits on tiles it requested moments before, keeps spinning.
// Bounded as mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}
// Non-blocking test of the phase: never suspends the thread.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity,
                                                long long limit_cycles = WAIT_LIMIT_CYCLES) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test(a, parity)) return true;  // (a phase already complete costs no suspension)
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_hint(a, parity, 20000u)) return true;
    if (clock64() - t0 > limit_cycles) return false;
  }
}

}  // namespace tc
}  // namespace gdn

namespace gdn {
namespace tc {

// ---- TMA tiled loads (tensor maps live in kernel parameter space) ---------------
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// shared-memory descriptor of an MN-major SW128 operand: the tile holds
// 64-element MN atoms of 128-byte rows along K; LBO is the distance between
// MN atoms, SBO the distance between 8-row K groups (1024 B)
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t mn_atom_stride) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(mn_atom_stride >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// D[128 x N] (+)= A * B^T where A (M = 128, K = 16 NK) is stored MN-major as a
// [128 (K) rows x 128 (M)] SW128 tile (NK = 4: its first 64 rows) and B is a
// K-major [N x 16 NK] SW128 tile
template <int NK = 8>
__device__ __forceinline__ void gemm_amn_k128(uint32_t tmem_d, uint32_t a_smem, uint32_t b_smem,
                                              int N, bool accumulate_first) {
  const uint32_t idesc = idesc_bf16(128, N) | (1u << 15);  // A is MN-major
  const uint64_t da0 = desc_sw128_mn(a_smem, 128u * 128u), db0 = desc_sw128(b_smem);  // (as gemm_k128)
#pragma unroll
  for (int k = 0; k < NK; ++k) {
    const uint64_t da = da0 + (((uint32_t)k * 2048u) >> 4);
    const uint32_t koff = (uint32_t)(k & 3) * 32u;
    const uint64_t db = db0 + (((uint32_t)(k >> 2) * (uint32_t)N * 128u + koff) >> 4);
    mma(tmem_d, da, db, idesc, (k > 0 || accumulate_first) ? 1u : 0u);
  }
}

// descriptor of a [K rows x 32] bf16 tile stored MN-major with 64-byte rows in the
// 64-byte swizzle (a tiled TMA load of 32 columns lands it): one 32-element
// atom along MN, 8-row groups of 512 bytes along K
__device__ __forceinline__ uint64_t desc_sw64_mn(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(512 >> 4) << 16;  // LBO (a single MN atom at N = 32)
  d |= (uint64_t)(512 >> 4) << 32;  // SBO: 8 K-rows of 64 bytes
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;           // 64-byte swizzle
  return d;
}
// D[128 x 32] = A * B where A (M = 128, K = 128) is stored MN-major as
// gemm_amn_k128 reads it and B (K = 128 rows, N = 32 columns) is the
// 64-byte-swizzled MN-major tile of desc_sw64_mn
__device__ __forceinline__ void gemm_amn_bmn64_k128(uint32_t tmem_d, uint32_t a_smem, uint32_t b_smem) {
  const uint32_t idesc = idesc_bf16(128, 32) | (1u << 15) | (1u << 16);  // A and B MN-major
  const uint64_t da0 = desc_sw128_mn(a_smem, 128u * 128u), db0 = desc_sw64_mn(b_smem);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    mma(tmem_d, da0 + (((uint32_t)k * 2048u) >> 4), db0 + (((uint32_t)k * 1024u) >> 4), idesc, k > 0 ? 1u : 0u);
}

// D[128 x 128] (+)= A * B where A is a K-major [128 x 128] SW128 tile and B
// (K = 128 rows, N = 128 columns) is stored MN-major: the [K rows x N] SW128
// tile as a tiled load of a row-major [K][N] matrix lands it (two 64-column
// atoms 16 KiB apart, 128-byte rows along K)
__device__ __forceinline__ void gemm_bmn_k128(uint32_t tmem_d, uint32_t a_smem, uint32_t b_smem,
                                              bool accumulate_first) {
  const uint32_t idesc = idesc_bf16(128, 128) | (1u << 16);  // B is MN-major
  const uint64_t da0 = desc_sw128(a_smem), db0 = desc_sw128_mn(b_smem, 128u * 128u);  // (as gemm_k128)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t koff = (uint32_t)(k & 3) * 32u;
    const uint64_t da = da0 + (((uint32_t)(k >> 2) * 128u * 128u + koff) >> 4);
    const uint64_t db = db0 + (((uint32_t)k * 2048u) >> 4);
    mma(tmem_d, da, db, idesc, (k > 0 || accumulate_first) ? 1u : 0u);
  }
}

// 32 fp32 columns into this thread's TMEM lane (complete after wait_st)
__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[128 x 128] (+)= A B^T-style product of two 128 x 128 SW128 operands, each
// either K-major (rows = M or N, 128-byte rows along K) or MN-major (rows =
// K, 128-byte rows along M or N: a row-major [K][M] matrix as a tiled load
// lands it)
__device__ __forceinline__ void gemm128(uint32_t tmem_d, uint32_t a_smem, bool a_mn, uint32_t b_smem,
                                        bool b_mn, bool accumulate_first) {
  const uint32_t idesc = idesc_bf16(128, 128) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
  const uint64_t da0 = a_mn ? desc_sw128_mn(a_smem, 128u * 128u) : desc_sw128(a_smem);  // (as gemm_k128)
  const uint64_t db0 = b_mn ? desc_sw128_mn(b_smem, 128u * 128u) : desc_sw128(b_smem);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t kmaj = (uint32_t)(k >> 2) * 128u * 128u + (uint32_t)(k & 3) * 32u;
    const uint64_t da = da0 + ((a_mn ? (uint32_t)k * 2048u : kmaj) >> 4);
    const uint64_t db = db0 + ((b_mn ? (uint32_t)k * 2048u : kmaj) >> 4);
    mma(tmem_d, da, db, idesc, (k > 0 || accumulate_first) ? 1u : 0u);
  }
}

// ---- TMA tiled stores (shared -> global), tracked by bulk async-groups -----------
// The shared source must have been written before a fence.proxy.async and a
// barrier; the issuing thread commits the group and later waits for it.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void tma_store_4d(const void* tmap, int x, int y, int z, int w, const void* src) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(tmap),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared sources of every committed store have been read (may be overwritten)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed store has completed
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// byte offset of the 16-byte chunk j (0..3) of row r in a [rows x 32] bf16 tile
// with the 64-byte swizzle (chunk j of row r sits at j ^ ((r / 2) % 4))
__device__ __forceinline__ uint32_t sw64_chunk(int r, int j) {
  return (uint32_t)(r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}

}  // namespace tc
}  // namespace gdn
