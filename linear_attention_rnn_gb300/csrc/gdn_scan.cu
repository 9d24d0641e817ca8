// gdn_scan.cu -- sequential walk of affine maps X <- A_i X (+ B_i).
//
// Serves two places:
//   * the cross-segment step of the two-pass segment scan ("Shard the
//     GatedDeltaNet sequence under ici_context_parallelism", description: an
//     exclusive prefix gives each stretch of chunks its incoming state):
//     h_in[0] = h0, h_in[s+1] = A_s h_in[s] + B_s (and, for the backward, the
//     same over the reversed segment order with the folded transposed maps);
//   * gdn_affine_compose, the inclusive prefix of (A, B) pairs under
//     (A2, B2) o (A1, B1) = (A2 A1, A2 B1 + B2) ("GatedDeltaNet does not
//     support ici_context_parallelism", composition law): the augmented state
//     [A_out | B_out] starts at [I | 0] and is pushed through the maps.
// One CTA walks one 16-column slice of the state (columns are independent).
// The products are fp32-accurate: A_i (fp32, read straight from global into
// mma fragments, one step ahead) and the state are both split into bf16
// hi + lo, and hi*hi + hi*lo + lo*hi is accumulated in fp32.
#include "gdn_kernels.cuh"

namespace gdn {

namespace {

constexpr int XC = 16;        // state columns per CTA
constexpr int LDX = XC + 8;   // bf16 row stride of the state image (48 bytes)

__global__ void __launch_bounds__(NTHREADS, 1) k_affine_walk(AffineWalkArgs a) {
  __shared__ __align__(16) bf16 Xh[HD * LDX];
  __shared__ __align__(16) bf16 Xl[HD * LDX];
  const int row = blockIdx.y;
  const int cs = blockIdx.x * XC;
  const bool inA = a.with_A && cs < HD;
  const int cB = a.with_A ? cs - HD : cs;  // column inside the B part
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int m0 = warp * 16;
  const int r0 = m0 + g4, r1 = r0 + 8;
  const long Astride = (long)HD * HD, Bstride = (long)HD * a.dv;

  float x[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = nt * 8 + 2 * t4 + e;
      if (inA) {
        x[nt][e] = (r0 == cs + col) ? 1.f : 0.f;
        x[nt][2 + e] = (r1 == cs + col) ? 1.f : 0.f;
      } else if (a.init) {
        const float* ip = a.init + (long)row * Bstride;
        x[nt][e] = ip[(long)r0 * a.dv + cB + col];
        x[nt][2 + e] = ip[(long)r1 * a.dv + cB + col];
      } else {
        x[nt][e] = 0.f;
        x[nt][2 + e] = 0.f;
      }
    }

  auto step_index = [&](int s) { return a.reverse ? a.n - 1 - s : s; };
  auto load_A = [&](int i, float2 (&f)[8][4]) {
    const float* Ap = a.A + ((long)row * a.n + i) * Astride;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c0 = ks * 16 + 2 * t4;
      f[ks][0] = *reinterpret_cast<const float2*>(Ap + (long)r0 * HD + c0);
      f[ks][1] = *reinterpret_cast<const float2*>(Ap + (long)r1 * HD + c0);
      f[ks][2] = *reinterpret_cast<const float2*>(Ap + (long)r0 * HD + c0 + 8);
      f[ks][3] = *reinterpret_cast<const float2*>(Ap + (long)r1 * HD + c0 + 8);
    }
  };
  auto store_state = [&](float* base) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(base + (long)r0 * (inA ? HD : a.dv) + col) = make_float2(x[nt][0], x[nt][1]);
      *reinterpret_cast<float2*>(base + (long)r1 * (inA ? HD : a.dv) + col) = make_float2(x[nt][2], x[nt][3]);
    }
  };
  auto out_ptr = [&](int i) -> float* {
    if (inA) return a.outA + ((long)row * a.n + i) * Astride + cs;
    return a.outB + ((long)row * a.n + i) * Bstride + cB;
  };

  float2 acur[8][4], anext[8][4];
  if (a.n > 0) load_A(step_index(0), acur);
  for (int s = 0; s < a.n; ++s) {
    const int i = step_index(s);
    if (a.exclusive) store_state(out_ptr(i));
    if (s + 1 < a.n) load_A(step_index(s + 1), anext);
    __syncthreads();  // previous step's readers of Xh/Xl are done
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = nt * 8 + 2 * t4;
      uint32_t h0, l0, h1, l1;
      split_bf16(x[nt][0], x[nt][1], h0, l0);
      split_bf16(x[nt][2], x[nt][3], h1, l1);
      *reinterpret_cast<uint32_t*>(Xh + r0 * LDX + col) = h0;
      *reinterpret_cast<uint32_t*>(Xl + r0 * LDX + col) = l0;
      *reinterpret_cast<uint32_t*>(Xh + r1 * LDX + col) = h1;
      *reinterpret_cast<uint32_t*>(Xl + r1 * LDX + col) = l1;
    }
    __syncthreads();
    float acc[2][4];
    if (!inA && a.Bv) {
      const float* Bp = a.Bv + ((long)row * a.n + i) * Bstride + cB;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = nt * 8 + 2 * t4;
        const float2 b0 = *reinterpret_cast<const float2*>(Bp + (long)r0 * a.dv + col);
        const float2 b1 = *reinterpret_cast<const float2*>(Bp + (long)r1 * a.dv + col);
        acc[nt][0] = b0.x;
        acc[nt][1] = b0.y;
        acc[nt][2] = b1.x;
        acc[nt][3] = b1.y;
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t ah[4], al[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) split_bf16(acur[ks][q].x, acur[ks][q].y, ah[q], al[q]);
      uint32_t bh[4], bl[4];
      ldb_kn(bh, Xh, LDX, ks * 16, 0, lane);
      ldb_kn(bl, Xl, LDX, ks * 16, 0, lane);
      mma16816(acc[0], ah, bh[0], bh[1]);
      mma16816(acc[1], ah, bh[2], bh[3]);
      mma16816(acc[0], ah, bl[0], bl[1]);
      mma16816(acc[1], ah, bl[2], bl[3]);
      mma16816(acc[0], al, bh[0], bh[1]);
      mma16816(acc[1], al, bh[2], bh[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[nt][e] = acc[nt][e];
    if (!a.exclusive) store_state(out_ptr(i));
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int q = 0; q < 4; ++q) acur[ks][q] = anext[ks][q];
  }
}

}  // namespace

cudaError_t launch_affine_walk(const AffineWalkArgs& a, cudaStream_t s) {
  const int ncols = (a.with_A ? HD : 0) + a.dv;
  dim3 grid(ncols / XC, a.batch);
  k_affine_walk<<<grid, NTHREADS, 0, s>>>(a);
  return cudaGetLastError();
}

// (A, B) = (I, 0) for n pairs: the fold of an empty stretch of chunks.
__global__ void k_identity_pairs(float* A, float* Bv, long n) {
  const long per = (long)HD * HD;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n * per; i += (long)gridDim.x * blockDim.x) {
    const long e = i % per;
    if (A) A[i] = (e / HD == e % HD) ? 1.f : 0.f;
    Bv[i] = 0.f;
  }
}

cudaError_t launch_identity_pairs(float* A, float* Bv, long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long total = n * HD * HD;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  k_identity_pairs<<<blocks, 256, 0, s>>>(A, Bv, n);
  return cudaGetLastError();
}

}  // namespace gdn
