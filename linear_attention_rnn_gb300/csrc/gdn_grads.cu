// gdn_grads.cu -- chunk-parallel gradients of the chunked gated delta rule.
//
// One CTA per (chunk c, value head j, batch row b), given the chunk's entering
// state h, the cotangent dh' of the state it leaves, Delta = u - w h and
// dDelta = P^T dO + k_g dh' (both stored by the two walks), and T.  Writing
// dV' = T^T dDelta, each line below reverses one line of the chunk forward:
//   u = T diag(beta) V        ->  dV = diag(beta) dV',  dbeta += rowsum(dV' * V)
//   w = T diag(beta gamma) K  ->  dK += -diag(beta gamma) dV' h^T, d(beta gamma) from it
//   T = (I + S)^-1            ->  dS = -(T^T dT T^T), strictly lower
//   S = tril(diag(beta) (K K^T * M), -1)  ->  dbeta, dK += dKK K + dKK^T K, dM
//   h' = gamma_C h + k_g^T Delta          ->  dK += diag(ef) Delta dh'^T, d ef, d gamma_C
//   O = diag(gamma) Q h + (Q K^T * M) Delta  ->  dQ, dK += dQK^T Q, d gamma, dM
// and the gate cotangent is the reverse cumsum of dG over the chunk.
// The analytic inverse backward dS = -(T^T dT T^T) ("Fuse the Gated Delta Net
// inter-chunk scan into a Pallas TPU kernel", section "Changes") is evaluated
// in the equal form dS = -dV' Delta^T: with dU = dDelta and dW = -dDelta h^T,
// dT = dDelta ((I+S) Delta)^T because (I+S) u = diag(beta) V and
// (I+S) w = diag(beta gamma) K, and T^T ... (I+S)^T T^T = I.
// dq and dk are written per value head in fp32; a second kernel sums the
// value heads of each key head.
#include "gdn_kernels.cuh"

namespace gdn {

namespace {

constexpr int TILE = CH * LDB;

struct GradSmem {
  bf16 t[6][TILE];
  float G[CH], gamma[CH], ef[CH], beta[CH], bg[CH];
  float dbeta[CH], dbg[CH], d_ef[CH], rowX[CH], dgamO[CH];
  float colX[8][CH];
  float red[8];
};

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}
// sum over the 8 row-groups g of a warp (lanes with equal t4)
__device__ __forceinline__ float rows_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

__device__ __forceinline__ void zero16(float (&acc)[16][4]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// acc[16 x 128] += A[rows m0..] (row-major tile) * B, B given as [n][k] tile
// (i.e. the product A X^T for row-major X), over k-steps [ks0, ks1).
__device__ __forceinline__ void gemm_rm_nk(float (&acc)[16][4], const bf16* A, const bf16* Bnk,
                                           int m0, int ks0, int ks1, int lane) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    if (ks < ks0 || ks >= ks1) continue;
    uint32_t af[4];
    lda_rm(af, A, LDB, m0, ks * 16, lane);
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t bb[4];
      ldb_nk(bb, Bnk, LDB, ks * 16, np * 16, lane);
      mma16816(acc[2 * np], af, bb[0], bb[1]);
      mma16816(acc[2 * np + 1], af, bb[2], bb[3]);
    }
  }
}
// acc += A * B with A row-major and B row-major [k][n].
__device__ __forceinline__ void gemm_rm_kn(float (&acc)[16][4], const bf16* A, const bf16* Bkn,
                                           int m0, int ks0, int ks1, int lane) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    if (ks < ks0 || ks >= ks1) continue;
    uint32_t af[4];
    lda_rm(af, A, LDB, m0, ks * 16, lane);
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t bb[4];
      ldb_kn(bb, Bkn, LDB, ks * 16, np * 16, lane);
      mma16816(acc[2 * np], af, bb[0], bb[1]);
      mma16816(acc[2 * np + 1], af, bb[2], bb[3]);
    }
  }
}
// acc += A^T * B with A stored row-major (so A^T is read transposed) and B row-major [k][n].
__device__ __forceinline__ void gemm_tr_kn(float (&acc)[16][4], const bf16* At, const bf16* Bkn,
                                           int m0, int ks0, int ks1, int lane) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    if (ks < ks0 || ks >= ks1) continue;
    uint32_t af[4];
    lda_tr(af, At, LDB, m0, ks * 16, lane);
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t bb[4];
      ldb_kn(bb, Bkn, LDB, ks * 16, np * 16, lane);
      mma16816(acc[2 * np], af, bb[0], bb[1]);
      mma16816(acc[2 * np + 1], af, bb[2], bb[3]);
    }
  }
}

__device__ __forceinline__ float2 ld_bf2(const bf16* p) {
  return unpack_bf16(*reinterpret_cast<const uint32_t*>(p));
}

__global__ void __launch_bounds__(NTHREADS, 1) k_grads(GradArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GradSmem& sm = *reinterpret_cast<GradSmem*>(smem_raw);
  bf16* t0 = sm.t[0];
  bf16* t1 = sm.t[1];
  bf16* t2 = sm.t[2];
  bf16* t3 = sm.t[3];
  bf16* t4 = sm.t[4];
  bf16* t5 = sm.t[5];
  const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g4 = lane >> 2, q4 = lane & 3;
  const int kh = j / (a.Hv / a.Hk);
  const int tk0 = c * CH;
  const int L = min(CH, a.T - tk0);
  const long bh = (long)b * a.Hv + j;
  const long cid = bh * a.NC + c;
  const long tokq = ((long)b * a.T + tk0) * a.Hk + kh;  // row 0 of the q/k tile
  const long tokv = ((long)b * a.T + tk0) * a.Hv + j;   // row 0 of the v/dO tile
  const int m0 = warp * 16;
  const int r0 = m0 + g4, r1 = r0 + 8;

  // group A: T, dDelta.  group B: h, Delta, K.
  tile_load_async(t0, a.Tb + cid * CH * CH, CH, CH, tid);
  tile_load_async(t1, a.ddelta + cid * CH * HD, HD, CH, tid);
  cp_async_commit();
  tile_load_async(t3, a.states + cid * HD * HD, HD, HD, tid);
  tile_load_async(t4, a.delta + cid * CH * HD, HD, CH, tid);
  tile_load_async(t5, a.k + tokq * HD, (long)a.Hk * HD, L, tid);
  cp_async_commit();
  if (tid < CH) {
    const long idx = tokv + (long)tid * a.Hv;
    sm.beta[tid] = tid < L ? a.beta[idx] : 0.f;
    sm.G[tid] = tid < L ? a.g[idx] : 0.f;
    sm.dbeta[tid] = 0.f;
    sm.rowX[tid] = 0.f;
  }
  for (int i = tid; i < 8 * CH; i += NTHREADS) (&sm.colX[0][0])[i] = 0.f;
  __syncthreads();
  if (warp == 0) {
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = sm.G[lane * 4 + i];
    warp_cumsum128(v, lane);
    const float Glast = __shfl_sync(0xffffffffu, v[3], 31);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      sm.G[r] = v[i];
      sm.gamma[r] = expf(v[i]);
      sm.ef[r] = expf(Glast - v[i]);
      sm.bg[r] = sm.beta[r] * sm.gamma[r];
    }
  }
  cp_async_wait<1>();
  __syncthreads();

  float acc[16][4], tmp[16][4];

  // ---- S1: dV' = T^T dDelta;  dv = beta dV';  dbeta += rowsum(dV' V) ---------
  zero16(tmp);
  gemm_tr_kn(tmp, t0, t1, m0, warp, 8, lane);  // T^T upper triangular: k >= m
  {
    const float b0 = sm.beta[r0], b1 = sm.beta[r1];
    float s0 = 0.f, s1 = 0.f;
    const bf16* vrow0 = a.v + (tokv + (long)r0 * a.Hv) * HD;
    const bf16* vrow1 = a.v + (tokv + (long)r1 * a.Hv) * HD;
    bf16* dv0 = a.dv + (tokv + (long)r0 * a.Hv) * HD;
    bf16* dv1 = a.dv + (tokv + (long)r1 * a.Hv) * HD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + 2 * q4;
      if (r0 < L) {
        const float2 vv = ld_bf2(vrow0 + col);
        s0 += tmp[nt][0] * vv.x + tmp[nt][1] * vv.y;
        *reinterpret_cast<uint32_t*>(dv0 + col) = pack_bf16(b0 * tmp[nt][0], b0 * tmp[nt][1]);
      }
      if (r1 < L) {
        const float2 vv = ld_bf2(vrow1 + col);
        s1 += tmp[nt][2] * vv.x + tmp[nt][3] * vv.y;
        *reinterpret_cast<uint32_t*>(dv1 + col) = pack_bf16(b1 * tmp[nt][2], b1 * tmp[nt][3]);
      }
      *reinterpret_cast<uint32_t*>(t2 + r0 * LDB + col) = pack_bf16(tmp[nt][0], tmp[nt][1]);
      *reinterpret_cast<uint32_t*>(t2 + r1 * LDB + col) = pack_bf16(tmp[nt][2], tmp[nt][3]);
    }
    s0 = quad_sum(s0);
    s1 = quad_sum(s1);
    if (q4 == 0) {
      sm.dbeta[r0] += s0;
      sm.dbeta[r1] += s1;
    }
  }
  __syncthreads();  // T, dDelta consumed; dV' complete
  // group C: dh' -> t1
  tile_load_async(t1, a.dstates + cid * HD * HD, HD, HD, tid);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();  // h, Delta, K ready

  // ---- S2: dK = -diag(beta gamma) dV' h^T;  dbg = rowsum(-(dV' h^T) K) --------
  zero16(tmp);
  gemm_rm_nk(tmp, t2, t3, m0, 0, 8, lane);
  {
    const float c0 = -sm.bg[r0], c1 = -sm.bg[r1];
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + 2 * q4;
      const float2 k0 = ld_bf2(t5 + r0 * LDB + col), k1 = ld_bf2(t5 + r1 * LDB + col);
      s0 -= tmp[nt][0] * k0.x + tmp[nt][1] * k0.y;
      s1 -= tmp[nt][2] * k1.x + tmp[nt][3] * k1.y;
      acc[nt][0] = c0 * tmp[nt][0];
      acc[nt][1] = c0 * tmp[nt][1];
      acc[nt][2] = c1 * tmp[nt][2];
      acc[nt][3] = c1 * tmp[nt][3];
    }
    s0 = quad_sum(s0);
    s1 = quad_sum(s1);
    if (q4 == 0) {
      sm.dbg[r0] = s0;
      sm.dbg[r1] = s1;
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // dh' ready

  // ---- S5: dK += diag(ef) Delta dh'^T;  d_ef = rowsum((Delta dh'^T) K);  <dh', h>
  zero16(tmp);
  gemm_rm_nk(tmp, t4, t1, m0, 0, 8, lane);
  {
    const float e0 = sm.ef[r0], e1 = sm.ef[r1];
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + 2 * q4;
      const float2 k0 = ld_bf2(t5 + r0 * LDB + col), k1 = ld_bf2(t5 + r1 * LDB + col);
      s0 += tmp[nt][0] * k0.x + tmp[nt][1] * k0.y;
      s1 += tmp[nt][2] * k1.x + tmp[nt][3] * k1.y;
      acc[nt][0] += e0 * tmp[nt][0];
      acc[nt][1] += e0 * tmp[nt][1];
      acc[nt][2] += e1 * tmp[nt][2];
      acc[nt][3] += e1 * tmp[nt][3];
    }
    s0 = quad_sum(s0);
    s1 = quad_sum(s1);
    if (q4 == 0) {
      sm.d_ef[r0] = s0;
      sm.d_ef[r1] = s1;
    }
    // <dh', h>: 128 x 128 elements, 64 per thread
    float d = 0.f;
    for (int i = tid; i < HD * HD / 2; i += NTHREADS) {
      const int r = (2 * i) >> 7, cc = (2 * i) & 127;
      const float2 x = ld_bf2(t1 + r * LDB + cc), y = ld_bf2(t3 + r * LDB + cc);
      d += x.x * y.x + x.y * y.y;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) sm.red[warp] = d;
  }
  __syncthreads();  // dh' consumed
  // group E: dO -> t1
  tile_load_async(t1, a.dO + tokv * HD, (long)a.Hv * HD, L, tid);
  cp_async_commit();

  // ---- S3: dS = -dV' Delta^T (strict lower);  KK;  dKK -> t0 --------------------
  {
    const float G0 = sm.G[r0], G1 = sm.G[r1], b0 = sm.beta[r0], b1 = sm.beta[r1];
    float db0 = 0.f, db1 = 0.f, x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      if (np > warp) continue;
      float ds[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float kk[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4], bb[4];
        lda_rm(af, t2, LDB, m0, ks * 16, lane);
        ldb_nk(bb, t4, LDB, ks * 16, np * 16, lane);
        mma16816(ds[0], af, bb[0], bb[1]);
        mma16816(ds[1], af, bb[2], bb[3]);
        lda_rm(af, t5, LDB, m0, ks * 16, lane);
        ldb_nk(bb, t5, LDB, ks * 16, np * 16, lane);
        mma16816(kk[0], af, bb[0], bb[1]);
        mma16816(kk[1], af, bb[2], bb[3]);
      }
      float cs[2][2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int s = np * 16 + h2 * 8 + 2 * q4 + e;
          const float Gs = sm.G[s];
          const float M0 = (s < r0) ? expf(G0 - Gs) : 0.f;
          const float M1 = (s < r1) ? expf(G1 - Gs) : 0.f;
          const float dS0 = -ds[h2][e] * (s < r0 ? 1.f : 0.f);
          const float dS1 = -ds[h2][2 + e] * (s < r1 ? 1.f : 0.f);
          const float KK0 = kk[h2][e], KK1 = kk[h2][2 + e];
          db0 += dS0 * KK0 * M0;
          db1 += dS1 * KK1 * M1;
          const float dkk0 = dS0 * b0 * M0, dkk1 = dS1 * b1 * M1;
          ds[h2][e] = dkk0;
          ds[h2][2 + e] = dkk1;
          const float X0 = dkk0 * KK0, X1 = dkk1 * KK1;
          x0 += X0;
          x1 += X1;
          cs[h2][e] = X0 + X1;
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int col = np * 16 + h2 * 8 + 2 * q4;
        *reinterpret_cast<uint32_t*>(t0 + r0 * LDB + col) = pack_bf16(ds[h2][0], ds[h2][1]);
        *reinterpret_cast<uint32_t*>(t0 + r1 * LDB + col) = pack_bf16(ds[h2][2], ds[h2][3]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = rows_sum(cs[h2][e]);
          if (g4 == 0) sm.colX[warp][col + e] += v;
        }
      }
    }
    // zero the strictly-upper tiles of dKK this warp did not write
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      if (np <= warp) continue;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int col = np * 16 + h2 * 8 + 2 * q4;
        *reinterpret_cast<uint32_t*>(t0 + r0 * LDB + col) = 0u;
        *reinterpret_cast<uint32_t*>(t0 + r1 * LDB + col) = 0u;
      }
    }
    db0 = quad_sum(db0);
    db1 = quad_sum(db1);
    x0 = quad_sum(x0);
    x1 = quad_sum(x1);
    if (q4 == 0) {
      sm.dbeta[r0] += db0;
      sm.dbeta[r1] += db1;
      sm.rowX[r0] += x0;
      sm.rowX[r1] += x1;
    }
  }
  __syncthreads();  // dV' consumed (t2 free); dKK complete
  // group D: Q -> t2
  tile_load_async(t2, a.q + tokq * HD, (long)a.Hk * HD, L, tid);
  cp_async_commit();

  // ---- S4: dK += dKK K + dKK^T K ----------------------------------------------
  gemm_rm_kn(acc, t0, t5, m0, 0, warp + 1, lane);
  gemm_tr_kn(acc, t0, t5, m0, warp, 8, lane);
  cp_async_wait<0>();
  __syncthreads();  // Q and dO ready; dKK consumed

  // ---- S6: dP = dO Delta^T;  QK;  dQK = dP * M (lower incl.) -> t0 ---------------
  {
    const float G0 = sm.G[r0], G1 = sm.G[r1];
    float x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      if (np > warp) continue;
      float dp[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float qk[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4], bb[4];
        lda_rm(af, t1, LDB, m0, ks * 16, lane);
        ldb_nk(bb, t4, LDB, ks * 16, np * 16, lane);
        mma16816(dp[0], af, bb[0], bb[1]);
        mma16816(dp[1], af, bb[2], bb[3]);
        lda_rm(af, t2, LDB, m0, ks * 16, lane);
        ldb_nk(bb, t5, LDB, ks * 16, np * 16, lane);
        mma16816(qk[0], af, bb[0], bb[1]);
        mma16816(qk[1], af, bb[2], bb[3]);
      }
      float cs[2][2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int s = np * 16 + h2 * 8 + 2 * q4 + e;
          const float Gs = sm.G[s];
          const float M0 = (s <= r0) ? expf(G0 - Gs) : 0.f;
          const float M1 = (s <= r1) ? expf(G1 - Gs) : 0.f;
          const float d0 = dp[h2][e] * M0, d1 = dp[h2][2 + e] * M1;
          dp[h2][e] = d0;
          dp[h2][2 + e] = d1;
          const float X0 = d0 * qk[h2][e], X1 = d1 * qk[h2][2 + e];
          x0 += X0;
          x1 += X1;
          cs[h2][e] = X0 + X1;
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int col = np * 16 + h2 * 8 + 2 * q4;
        *reinterpret_cast<uint32_t*>(t0 + r0 * LDB + col) = pack_bf16(dp[h2][0], dp[h2][1]);
        *reinterpret_cast<uint32_t*>(t0 + r1 * LDB + col) = pack_bf16(dp[h2][2], dp[h2][3]);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = rows_sum(cs[h2][e]);
          if (g4 == 0) sm.colX[warp][col + e] += v;
        }
      }
    }
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      if (np <= warp) continue;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int col = np * 16 + h2 * 8 + 2 * q4;
        *reinterpret_cast<uint32_t*>(t0 + r0 * LDB + col) = 0u;
        *reinterpret_cast<uint32_t*>(t0 + r1 * LDB + col) = 0u;
      }
    }
    x0 = quad_sum(x0);
    x1 = quad_sum(x1);
    if (q4 == 0) {
      sm.rowX[r0] += x0;
      sm.rowX[r1] += x1;
    }
  }
  __syncthreads();  // dQK complete

  // ---- S7: dK += dQK^T Q  -> dk (per value head, fp32) ---------------------------
  gemm_tr_kn(acc, t0, t2, m0, warp, 8, lane);
  {
    float* d0 = a.dk_part + (tokv + (long)r0 * a.Hv) * HD;
    float* d1 = a.dk_part + (tokv + (long)r1 * a.Hv) * HD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + 2 * q4;
      if (r0 < L) *reinterpret_cast<float2*>(d0 + col) = make_float2(acc[nt][0], acc[nt][1]);
      if (r1 < L) *reinterpret_cast<float2*>(d1 + col) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }

  // ---- S8: dQ = diag(gamma) dO h^T + dQK K;  dgamma_O = rowsum(Q * (dO h^T)) ---
  zero16(acc);
  gemm_rm_nk(acc, t1, t3, m0, 0, 8, lane);
  {
    const float gm0 = sm.gamma[r0], gm1 = sm.gamma[r1];
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + 2 * q4;
      const float2 q0 = ld_bf2(t2 + r0 * LDB + col), q1 = ld_bf2(t2 + r1 * LDB + col);
      s0 += acc[nt][0] * q0.x + acc[nt][1] * q0.y;
      s1 += acc[nt][2] * q1.x + acc[nt][3] * q1.y;
      acc[nt][0] *= gm0;
      acc[nt][1] *= gm0;
      acc[nt][2] *= gm1;
      acc[nt][3] *= gm1;
    }
    s0 = quad_sum(s0);
    s1 = quad_sum(s1);
    if (q4 == 0) {
      sm.dgamO[r0] = s0;
      sm.dgamO[r1] = s1;
    }
  }
  gemm_rm_kn(acc, t0, t5, m0, 0, warp + 1, lane);
  {
    float* d0 = a.dq_part + (tokv + (long)r0 * a.Hv) * HD;
    float* d1 = a.dq_part + (tokv + (long)r1 * a.Hv) * HD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int col = nt * 8 + 2 * q4;
      if (r0 < L) *reinterpret_cast<float2*>(d0 + col) = make_float2(acc[nt][0], acc[nt][1]);
      if (r1 < L) *reinterpret_cast<float2*>(d1 + col) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();  // all row/column vectors complete

  // ---- S9: gate cotangents -------------------------------------------------------
  if (warp == 0) {
    float dgC = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) dgC += sm.red[w];
    float sum_def = 0.f;
    float dG[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      float col = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) col += sm.colX[w][r];
      const float de = sm.d_ef[r] * sm.ef[r];
      sum_def += de;
      const float dgam = sm.dgamO[r] + sm.beta[r] * sm.dbg[r];
      dG[i] = sm.gamma[r] * dgam + sm.rowX[r] - col - de;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum_def += __shfl_xor_sync(0xffffffffu, sum_def, off);
    if (lane == 31) dG[3] += sm.gamma[CH - 1] * dgC + sum_def;  // row C-1: gamma_C = gamma[C-1]
    // reverse inclusive cumsum over the 128 rows: dg_s = sum_{r >= s} dG_r
    float tot = dG[0] + dG[1] + dG[2] + dG[3];
    float incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += o;
    }
    float run = incl - tot;  // sum over lanes > lane
    float dg[4];
#pragma unroll
    for (int i = 3; i >= 0; --i) {
      run += dG[i];
      dg[i] = run;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      if (r < L) {
        a.dg[tokv + (long)r * a.Hv] = dg[i];
        a.dbeta[tokv + (long)r * a.Hv] = sm.dbeta[r] + sm.gamma[r] * sm.dbg[r];
      }
    }
  }
}

__global__ void k_reduce_dqdk(const float* __restrict__ dqp, const float* __restrict__ dkp,
                              bf16* __restrict__ dq, bf16* __restrict__ dk, long tokens, int Hk,
                              int Hv) {
  const int group = Hv / Hk;
  const long n4 = tokens * Hk * (HD / 4);
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n4; i += (long)gridDim.x * blockDim.x) {
    const long tk = i / (Hk * (HD / 4));
    const int rem = (int)(i % (Hk * (HD / 4)));
    const int kh = rem / (HD / 4), c4 = (rem % (HD / 4)) * 4;
    float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
    for (int r = 0; r < group; ++r) {
      const long src = (tk * Hv + kh * group + r) * HD + c4;
      const float4 x = *reinterpret_cast<const float4*>(dqp + src);
      const float4 y = *reinterpret_cast<const float4*>(dkp + src);
      sq.x += x.x; sq.y += x.y; sq.z += x.z; sq.w += x.w;
      sk.x += y.x; sk.y += y.y; sk.z += y.z; sk.w += y.w;
    }
    const long dst = (tk * Hk + kh) * HD + c4;
    uint2 oq, ok;
    oq.x = pack_bf16(sq.x, sq.y);
    oq.y = pack_bf16(sq.z, sq.w);
    ok.x = pack_bf16(sk.x, sk.y);
    ok.y = pack_bf16(sk.z, sk.w);
    *reinterpret_cast<uint2*>(dq + dst) = oq;
    *reinterpret_cast<uint2*>(dk + dst) = ok;
  }
}

}  // namespace

size_t grad_smem_bytes() { return sizeof(GradSmem); }

cudaError_t launch_grads(const GradArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(GradSmem);
  cudaError_t e = cudaFuncSetAttribute(k_grads, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_grads<<<dim3(a.NC, a.Hv, a.B), NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reduce_dqdk(const float* dq_part, const float* dk_part, bf16* dq, bf16* dk,
                               long tokens, int Hk, int Hv, cudaStream_t s) {
  const long n4 = tokens * Hk * (HD / 4);
  if (n4 == 0) return cudaSuccess;
  long blocks = (n4 + 255) / 256;
  if (blocks > 152L * 16) blocks = 152L * 16;
  k_reduce_dqdk<<<(int)blocks, 256, 0, s>>>(dq_part, dk_part, dq, dk, tokens, Hk, Hv);
  return cudaGetLastError();
}

}  // namespace gdn
