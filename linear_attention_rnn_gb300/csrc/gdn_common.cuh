// gdn_common.cuh -- shared device helpers of the GB300 gated-delta-rule kernels.
//
// Tiles are 128 x 128 (chunk rows x head dim).  bf16 tiles live in shared
// memory with a padded row stride of LDB elements (272 bytes) so that the 8
// row addresses of every ldmatrix phase fall in distinct bank groups.
// Warp-level tensor-core products use mma.sync m16n8k16 (bf16 in, fp32
// accumulate); fragment layouts follow the PTX ISA description of that shape:
//   A (16x16, row):  a0 = (g, 2t..2t+1)   a1 = (g+8, 2t..)   a2 = (g, 2t+8..)  a3 = (g+8, 2t+8..)
//   B (16x8, col):   b0 = (k 2t..2t+1, n g)   b1 = (k 2t+8..2t+9, n g)
//   C (16x8, f32):   c0,c1 = (g, 2t..2t+1)    c2,c3 = (g+8, 2t..2t+1)
// with g = lane / 4 and t = lane % 4.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int CH = 128;        // chunk rows
constexpr int HD = 128;        // head dim (d_k = d_v)
constexpr int LDB = HD + 8;    // padded bf16 row stride of a 128-wide tile (elements)
constexpr int NTHREADS = 256;  // 8 warps; warp w owns rows 16w..16w+15 of a 128-row product
constexpr int SL = 32;         // state-column slice width of the sequential walks
constexpr int LDS_ = SL + 8;   // padded bf16 row stride of a 32-wide slice tile (80 bytes)

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared async copy; when !valid the destination is zero-filled
// and no global byte is read (src must still be a mapped address).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}
// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): the two-term split used
// for fp32-accurate products (hi*hi + hi*lo + lo*hi, fp32 accumulate).
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// ---- fragment loaders from bf16 shared tiles -------------------------------
// A[m][k] stored row-major (m rows, stride ld): 16x16 block at (m0, k0).
__device__ __forceinline__ void lda_rm(uint32_t (&a)[4], const bf16* base, int ld, int m0,
                                       int k0, int lane) {
  ldsm_x4(a, base + (m0 + (lane & 15)) * ld + k0 + ((lane >> 4) << 3));
}
// A[m][k] stored transposed as [k][m] (stride ld): 16x16 block at (m0, k0).
__device__ __forceinline__ void lda_tr(uint32_t (&a)[4], const bf16* base, int ld, int m0,
                                       int k0, int lane) {
  const int i = lane >> 3, r = lane & 7;
  ldsm_x4_t(a, base + (k0 + ((i >> 1) << 3) + r) * ld + m0 + ((i & 1) << 3));
}
// B[k][n] stored row-major as [k][n]: two n-tiles (n0..n0+7, n0+8..n0+15) of k0..k0+15.
// b[0],b[1] = (b0,b1) of the first n-tile, b[2],b[3] of the second.
__device__ __forceinline__ void ldb_kn(uint32_t (&b)[4], const bf16* base, int ld, int k0,
                                       int n0, int lane) {
  ldsm_x4_t(b, base + (k0 + (lane & 15)) * ld + n0 + ((lane >> 4) << 3));
}
// B[k][n] stored as [n][k] (e.g. B = X^T with X row-major): same output order.
__device__ __forceinline__ void ldb_nk(uint32_t (&b)[4], const bf16* base, int ld, int k0,
                                       int n0, int lane) {
  const int i = lane >> 3, r = lane & 7;
  ldsm_x4(b, base + (n0 + ((i >> 1) << 3) + r) * ld + k0 + ((i & 1) << 3));
}

// ---- tile copies ---------------------------------------------------------------
// Copy `rows` valid rows of a [128 x 128] bf16 tile from global (row stride
// gstride elements) into a padded shared tile; rows >= rows are zero-filled.
__device__ __forceinline__ void tile_load_async(bf16* s, const bf16* g, long gstride, int rows,
                                                int tid) {
#pragma unroll
  for (int i = 0; i < (CH * HD / 8) / NTHREADS; ++i) {
    const int idx = tid + i * NTHREADS;
    const int r = idx >> 4, c8 = (idx & 15) << 3;
    const bool ok = r < rows;
    cp_async16(s + r * LDB + c8, g + (ok ? (long)r * gstride + c8 : 0), ok);
  }
}
// Same for a [128 x 32] column slice starting at column col0 of a global tile.
__device__ __forceinline__ void slice_load_async(bf16* s, const bf16* g, long gstride, int rows,
                                                 int tid) {
  // 128 rows x 4 chunks of 8 elements = 512 copies, 2 per thread
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = tid + i * NTHREADS;
    const int r = idx >> 2, c8 = (idx & 3) << 3;
    const bool ok = r < rows;
    cp_async16(s + r * LDS_ + c8, g + (ok ? (long)r * gstride + c8 : 0), ok);
  }
}

// ---- XOR-swizzled [rows x 128] bf16 tiles (256-byte rows, no padding) ----------
// The 16-byte chunk j of row r sits at chunk position j ^ (r & 7), so the 8 row
// addresses of every ldmatrix phase fall in 8 distinct bank groups.
__device__ __forceinline__ const bf16* swz(const bf16* base, int r, int j) {
  return base + r * HD + ((j ^ (r & 7)) << 3);
}
__device__ __forceinline__ bf16* swz(bf16* base, int r, int j) {
  return base + r * HD + ((j ^ (r & 7)) << 3);
}
__device__ __forceinline__ void lda_rm_s(uint32_t (&a)[4], const bf16* base, int m0, int k0,
                                         int lane) {
  ldsm_x4(a, swz(base, m0 + (lane & 15), (k0 >> 3) + (lane >> 4)));
}
__device__ __forceinline__ void lda_tr_s(uint32_t (&a)[4], const bf16* base, int m0, int k0,
                                         int lane) {
  const int i = lane >> 3, r = lane & 7;
  ldsm_x4_t(a, swz(base, k0 + ((i >> 1) << 3) + r, (m0 >> 3) + (i & 1)));
}
__device__ __forceinline__ void ldb_kn_s(uint32_t (&b)[4], const bf16* base, int k0, int n0,
                                         int lane) {
  ldsm_x4_t(b, swz(base, k0 + (lane & 15), (n0 >> 3) + (lane >> 4)));
}
__device__ __forceinline__ void ldb_nk_s(uint32_t (&b)[4], const bf16* base, int k0, int n0,
                                         int lane) {
  const int i = lane >> 3, r = lane & 7;
  ldsm_x4(b, swz(base, n0 + ((i >> 1) << 3) + r, (k0 >> 3) + (i & 1)));
}
// rows [0, rows) of a [128 x 128] global tile (row stride gstride) into a
// swizzled shared tile; rows past `rows` are zero-filled
__device__ __forceinline__ void tile_load_async_s(bf16* s, const bf16* g, long gstride, int rows,
                                                  int tid, int nthreads) {
  for (int idx = tid; idx < CH * 16; idx += nthreads) {
    const int r = idx >> 4, j = idx & 15;
    const bool ok = r < rows;
    cp_async16(swz(s, r, j), g + (ok ? (long)r * gstride + j * 8 : 0), ok);
  }
}
// cp.async.wait_group with a run-time count (0..7)
__device__ __forceinline__ void cp_async_wait_n(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
  }
}

// ---- bulk async copies completing on transaction-count mbarriers ---------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Waits for the phase of the given parity; gives up after a bounded number of
// polls and returns false.
__device__ __forceinline__ bool mbar_wait_parity(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  for (int it = 0; it < (1 << 22); ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Rows [0, rows) of a [128 x 128] bf16 global tile (row stride gstride) into
// a padded shared tile, one 256-byte bulk copy per row, issued by the 32
// lanes of one warp; rows past `rows` are cleared with ordinary stores (the
// caller orders them with a CTA barrier).  Completes rows * 256 bytes on bar.
__device__ __forceinline__ void tile_bulk_rows(bf16* s, const bf16* g, long gstride, int rows,
                                               uint64_t* bar, int lane) {
  for (int r = lane; r < CH; r += 32) {
    if (r < rows) {
      bulk_g2s(s + r * LDB, g + (long)r * gstride, HD * sizeof(bf16), bar);
    } else {
#pragma unroll
      for (int c8 = 0; c8 < HD; c8 += 8) *reinterpret_cast<uint4*>(s + r * LDB + c8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}
// Same for a [128 x 32] column slice (64-byte rows) into a padded slice tile.
__device__ __forceinline__ void slice_bulk_rows(bf16* s, const bf16* g, long gstride, int rows,
                                                uint64_t* bar, int lane) {
  for (int r = lane; r < CH; r += 32) {
    if (r < rows) {
      bulk_g2s(s + r * LDS_, g + (long)r * gstride, SL * sizeof(bf16), bar);
    } else {
#pragma unroll
      for (int c8 = 0; c8 < SL; c8 += 8) *reinterpret_cast<uint4*>(s + r * LDS_ + c8) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Inclusive prefix sum over the 128 values held 4-per-lane by one warp
// (lane l holds rows 4l..4l+3 in v[0..3]).
__device__ __forceinline__ void warp_cumsum128(float (&v)[4], int lane) {
  v[1] += v[0];
  v[2] += v[1];
  v[3] += v[2];
  float run = v[3];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float o = __shfl_up_sync(0xffffffffu, run, off);
    if (lane >= off) run += o;
  }
  const float excl = run - v[3];
  v[0] += excl;
  v[1] += excl;
  v[2] += excl;
  v[3] += excl;
}

}  // namespace gdn
