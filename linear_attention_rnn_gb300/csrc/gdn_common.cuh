// gdn_common.cuh -- shared device helpers of the GB300 gated-delta-rule kernels.
//
// Tiles are 128 x 128 (chunk rows x head dim).  The large products run on the
// tcgen05 tensor cores (gdn_tc05.cuh); the small fp32-accurate ones (the
// ladder of the triangular inverse, the segment prefix) use warp-level
// mma.sync m16n8k16 (bf16 in, fp32 accumulate), whose fragment layouts follow
// the PTX ISA description of that shape:
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
constexpr int NTHREADS = 256;  // 8 warps (prep and gradient kernels)
constexpr int SL = 32;         // state-column slice width of the sequential walks

typedef __nv_bfloat16 bf16;

// Programmatic dependent launch.  A kernel launched with the programmatic
// serialization attribute may start while the kernel before it in the stream
// still runs; pdl_wait() returns once that kernel has completed and its
// memory is visible (at once when the kernel was launched normally).  Every
// kernel of this library waits before it reads anything the kernel before it
// may write and before it writes anything, and only then lets its own
// dependents start (pdl_release), so that when a kernel starts, every kernel
// before its immediate predecessor has completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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

// Predicated read-only global loads straight into the destination registers:
// with pred false nothing is read and the registers keep their values.  A plain
// `v = pred ? *p : 0` merges the loaded value into v with an instruction that
// waits for the load where it is issued; these leave the wait to the first real
// use of v.  p must point to readable memory whenever pred is true.
__device__ __forceinline__ void ld_pred_v4(uint4& v, const void* p, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}\n"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "l"(p), "r"((int)pred));
}
__device__ __forceinline__ void ld_pred_f32(float& v, const float* p, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
      "@q ld.global.nc.f32 %0, [%1];\n\t}\n"
      : "+f"(v)
      : "l"(p), "r"((int)pred));
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
// B[k][n] stored row-major as [k][n]: two n-tiles (n0..n0+7, n0+8..n0+15) of k0..k0+15.
// b[0],b[1] = (b0,b1) of the first n-tile, b[2],b[3] of the second.
__device__ __forceinline__ void ldb_kn(uint32_t (&b)[4], const bf16* base, int ld, int k0,
                                       int n0, int lane) {
  ldsm_x4_t(b, base + (k0 + (lane & 15)) * ld + n0 + ((lane >> 4) << 3));
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
// A[m][k] stored row-major in a swizzled tile: 16x16 block at (m0, k0).
__device__ __forceinline__ void lda_rm_s(uint32_t (&a)[4], const bf16* base, int m0, int k0,
                                         int lane) {
  ldsm_x4(a, swz(base, m0 + (lane & 15), (k0 >> 3) + (lane >> 4)));
}
// B[k][n] stored row-major in a swizzled tile: same output order as ldb_kn.
__device__ __forceinline__ void ldb_kn_s(uint32_t (&b)[4], const bf16* base, int k0, int n0,
                                         int lane) {
  ldsm_x4_t(b, swz(base, k0 + (lane & 15), (n0 >> 3) + (lane >> 4)));
}

// Inclusive prefix sum over the 128 values held 4-per-lane by one warp
// (lane l holds rows 4l..4l+3 in v[0..3]).
// (split64: two independent scans, rows 0..63 and 64..127, i.e. lanes 0-15 and 16-31)
__device__ __forceinline__ void warp_cumsum128(float (&v)[4], int lane, bool split64 = false) {
  v[1] += v[0];
  v[2] += v[1];
  v[3] += v[2];
  float run = v[3];
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float o = __shfl_up_sync(0xffffffffu, run, off);
    if (lane >= off && (!split64 || ((lane ^ (lane - off)) & 16) == 0)) run += o;
  }
  const float excl = run - v[3];
  v[0] += excl;
  v[1] += excl;
  v[2] += excl;
  v[3] += excl;
}

// Gate activations, applied where the kernels load the gates when the caller
// passes logits (logits != 0): beta = sigmoid(b) and g = -softplus(a), the
// decay exp(g) = 1 / (1 + exp(a)).  softplus(a) = max(a, 0) + log1p(exp(-|a|)).
__device__ __forceinline__ float act_g(float a, int logits) {
  return logits ? -(fmaxf(a, 0.f) + log1pf(expf(-fabsf(a)))) : a;
}
__device__ __forceinline__ float act_beta(float b, int logits) {
  return logits ? 1.f / (1.f + expf(-b)) : b;
}

}  // namespace gdn

