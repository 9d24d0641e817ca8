// gdn_prep.cu -- per-chunk UT/WY preparation of the chunked gated delta rule.
//
// One CTA per (chunk c, value head j, batch row b) computes, for the 128 rows
// of its chunk (zero-padded past T with g = 0, beta = 0):
//   gates   G = chunk-local cumsum of g, gamma = exp(G)
//   S       = tril(diag(beta) (K K^T * M), -1),  M_rs = exp(G_r - G_s) (s <= r,
//             exponent masked before the exp so nothing overflows)
//   P       = (Q K^T) * M including the diagonal          (for the output)
//   T       = (I + S)^-1 by the blockwise doubling ladder
//   w       = T diag(beta gamma) K,   u = T diag(beta) V
// The ladder ("Fuse the Gated Delta Net inter-chunk scan into a Pallas TPU
// kernel", section "Changes", triangular inversion kernel): with X the
// inverse of I + S on its diagonal blocks of size b, the inverse on blocks of
// size 2b is X - X S_l X, where S_l is the lower-left b x b block of each
// 2b x 2b diagonal block.  Here the 16 x 16 diagonal blocks are inverted
// exactly in fp32 by forward substitution (one warp each, the ladder's
// levels b = 1..8 folded into one exact step) and the levels b = 16, 32, 64
// run on the tensor cores with two-term bf16 operand splitting
// (hi*hi + hi*lo + lo*hi, fp32 accumulate), which keeps T at fp32-like accuracy.
// The 2b-level update only touches the lower-left block: X - X S_l X there is
// -X_D S_C X_A, computed as Y = S_C X_A, then -X_D Y.
#include "gdn_kernels.cuh"

namespace gdn {

namespace {

constexpr int LDF = HD + 8;  // fp32 row stride of the S/T tile
constexpr int LDY = 64 + 4;  // fp32 row stride of the ladder scratch

struct PrepSmem {
  bf16 K[CH * LDB];
  bf16 QV[CH * LDB];  // Q, then V
  float ST[CH * LDF]; // S, overwritten in place by T
  float Y[64 * LDY];
  float g[CH], beta[CH], G[CH], gamma[CH], bg[CH];
};

// 16x16 fp32 block (row-major, stride lda) times 16x8 fp32 block ([k][n],
// stride ldb), fp32-accurate via two-term bf16 splitting.
__device__ __forceinline__ void mma_split(float (&d)[4], const float* pa, int lda,
                                          const float* pb, int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const float2 x0 = *reinterpret_cast<const float2*>(pa + g * lda + 2 * t);
  const float2 x1 = *reinterpret_cast<const float2*>(pa + (g + 8) * lda + 2 * t);
  const float2 x2 = *reinterpret_cast<const float2*>(pa + g * lda + 2 * t + 8);
  const float2 x3 = *reinterpret_cast<const float2*>(pa + (g + 8) * lda + 2 * t + 8);
  uint32_t ah[4], al[4];
  split_bf16(x0.x, x0.y, ah[0], al[0]);
  split_bf16(x1.x, x1.y, ah[1], al[1]);
  split_bf16(x2.x, x2.y, ah[2], al[2]);
  split_bf16(x3.x, x3.y, ah[3], al[3]);
  uint32_t bh0, bl0, bh1, bl1;
  split_bf16(pb[(2 * t) * ldb + g], pb[(2 * t + 1) * ldb + g], bh0, bl0);
  split_bf16(pb[(2 * t + 8) * ldb + g], pb[(2 * t + 9) * ldb + g], bh1, bl1);
  mma16816(d, ah, bh0, bh1);
  mma16816(d, ah, bl0, bl1);
  mma16816(d, al, bh0, bh1);
}

// A fragment (16x16 at rows m0, cols k0) from the fp32 T tile with the column
// scale s[k] applied, rounded to bf16.
__device__ __forceinline__ void lda_f32_colscaled(uint32_t (&a)[4], const float* base, int m0,
                                                  int k0, const float* s, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int c0 = k0 + 2 * t, c1 = c0 + 8;
  const float s00 = s[c0], s01 = s[c0 + 1], s10 = s[c1], s11 = s[c1 + 1];
  const float* r0 = base + (m0 + g) * LDF;
  const float* r1 = base + (m0 + g + 8) * LDF;
  a[0] = pack_bf16(r0[c0] * s00, r0[c0 + 1] * s01);
  a[1] = pack_bf16(r1[c0] * s00, r1[c0 + 1] * s01);
  a[2] = pack_bf16(r0[c1] * s10, r0[c1 + 1] * s11);
  a[3] = pack_bf16(r1[c1] * s10, r1[c1 + 1] * s11);
}

// Store a warp's 16 x 128 fp32 accumulator block (rows m0..m0+15) as bf16.
__device__ __forceinline__ void store_rows_bf16(bf16* dst, int ld, int m0, const float (&acc)[16][4],
                                                int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int col = nt * 8 + 2 * t;
    *reinterpret_cast<uint32_t*>(dst + (long)(m0 + g) * ld + col) = pack_bf16(acc[nt][0], acc[nt][1]);
    *reinterpret_cast<uint32_t*>(dst + (long)(m0 + g + 8) * ld + col) =
        pack_bf16(acc[nt][2], acc[nt][3]);
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) k_prep(PrepArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
  const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int kh = j / (a.Hv / a.Hk);
  const int t0 = c * CH;
  const int L = min(CH, a.T - t0);
  const long tokstride = (long)a.Hk * HD;
  const long bh = (long)b * a.Hv + j;
  const long chunk_id = bh * a.NC + c;
  const bf16* kgl = a.k + (((long)b * a.T + t0) * a.Hk + kh) * HD;
  const bf16* qgl = a.q + (((long)b * a.T + t0) * a.Hk + kh) * HD;
  const bf16* vgl = a.v + (((long)b * a.T + t0) * a.Hv + j) * HD;
  const bool needP = a.P != nullptr;
  const bool needU = a.U != nullptr;

  tile_load_async(sm.K, kgl, tokstride, L, tid);
  if (needP) tile_load_async(sm.QV, qgl, tokstride, L, tid);
  cp_async_commit();
  if (tid < CH) {
    const long idx = ((long)b * a.T + t0 + tid) * a.Hv + j;
    sm.g[tid] = tid < L ? a.g[idx] : 0.f;
    sm.beta[tid] = tid < L ? a.beta[idx] : 0.f;
  }
  __syncthreads();
  if (warp == 0) {
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = sm.g[lane * 4 + i];
    warp_cumsum128(v, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      const float gm = expf(v[i]);
      sm.G[r] = v[i];
      sm.gamma[r] = gm;
      sm.bg[r] = sm.beta[r] * gm;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  const int m0 = warp * 16;
  const int r0 = m0 + g4, r1 = r0 + 8;
  float acc[16][4];

  // ---- S = tril(diag(beta) (K K^T * M), -1) --------------------------------
  {
    uint32_t af[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) lda_rm(af[ks], sm.K, LDB, m0, ks * 16, lane);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      if (np <= warp) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t bb[4];
          ldb_nk(bb, sm.K, LDB, ks * 16, np * 16, lane);
          mma16816(acc[2 * np], af[ks], bb[0], bb[1]);
          mma16816(acc[2 * np + 1], af[ks], bb[2], bb[3]);
        }
      }
    }
    const float G0 = sm.G[r0], G1 = sm.G[r1], b0 = sm.beta[r0], b1 = sm.beta[r1];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int s = nt * 8 + 2 * t4 + e;
        const float Gs = sm.G[s];
        const float v0 = (s < r0) ? b0 * acc[nt][e] * expf(G0 - Gs) : 0.f;
        const float v1 = (s < r1) ? b1 * acc[nt][2 + e] * expf(G1 - Gs) : 0.f;
        sm.ST[r0 * LDF + s] = v0;
        sm.ST[r1 * LDF + s] = v1;
      }
    }
  }
  // ---- P = (Q K^T) * M, diagonal included ------------------------------------
  if (needP) {
    uint32_t af[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) lda_rm(af[ks], sm.QV, LDB, m0, ks * 16, lane);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      if (np <= warp) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t bb[4];
          ldb_nk(bb, sm.K, LDB, ks * 16, np * 16, lane);
          mma16816(acc[2 * np], af[ks], bb[0], bb[1]);
          mma16816(acc[2 * np + 1], af[ks], bb[2], bb[3]);
        }
      }
    }
    const float G0 = sm.G[r0], G1 = sm.G[r1];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int s = nt * 8 + 2 * t4 + e;
        const float Gs = sm.G[s];
        acc[nt][e] = (s <= r0) ? acc[nt][e] * expf(G0 - Gs) : 0.f;
        acc[nt][2 + e] = (s <= r1) ? acc[nt][2 + e] * expf(G1 - Gs) : 0.f;
      }
    }
    store_rows_bf16(a.P + chunk_id * CH * CH, CH, m0, acc, lane);
  }
  __syncthreads();  // Q no longer needed; S complete
  if (needU) {
    tile_load_async(sm.QV, vgl, (long)a.Hv * HD, L, tid);
  }
  cp_async_commit();

  if (a.S_dbg) {
    float* dst = a.S_dbg + chunk_id * CH * CH;
    for (int i = tid; i < CH * CH; i += NTHREADS) dst[i] = sm.ST[(i >> 7) * LDF + (i & 127)];
  }
  __syncthreads();  // debug copy done before S is overwritten

  // ---- T = (I + S)^-1 --------------------------------------------------------
  // (1) 16x16 diagonal blocks, exact forward substitution, one warp per block.
  {
    const int base = 16 * warp;
    for (int i = 0; i < 16; ++i) {
      float* row = &sm.ST[(base + i) * LDF + base];
      const float srow = (lane < 16) ? row[lane] : 0.f;
      __syncwarp();
      float x = (lane == i) ? 1.f : 0.f;
      for (int s = 0; s < i; ++s) {
        const float Sis = __shfl_sync(0xffffffffu, srow, s);
        const float Tsj = (lane < 16) ? sm.ST[(base + s) * LDF + base + lane] : 0.f;
        x -= Sis * Tsj;
      }
      if (lane < 16) row[lane] = x;
      __syncwarp();
    }
  }
  __syncthreads();
  // (2) ladder levels b = 16, 32, 64 on the lower-left blocks.
  for (int bs = 16; bs < CH; bs *= 2) {
    const int tiles_m = bs / 16, tiles_n = bs / 8;
    const int per_pair = tiles_m * tiles_n;
    const int ntiles = (CH / (2 * bs)) * per_pair;
    for (int tile = warp; tile < ntiles; tile += 8) {
      const int p = tile / per_pair, rem = tile % per_pair;
      const int tm = rem / tiles_n, tn = rem % tiles_n;
      const int s0 = p * 2 * bs;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = 0; k0 < bs; k0 += 16)
        mma_split(d, &sm.ST[(s0 + bs + 16 * tm) * LDF + s0 + k0], LDF,
                  &sm.ST[(s0 + k0) * LDF + s0 + 8 * tn], LDF, lane);
      float* y0 = &sm.Y[(p * bs + 16 * tm + g4) * LDY + 8 * tn + 2 * t4];
      y0[0] = d[0];
      y0[1] = d[1];
      y0[8 * LDY] = d[2];
      y0[8 * LDY + 1] = d[3];
    }
    __syncthreads();
    for (int tile = warp; tile < ntiles; tile += 8) {
      const int p = tile / per_pair, rem = tile % per_pair;
      const int tm = rem / tiles_n, tn = rem % tiles_n;
      const int s0 = p * 2 * bs;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = 0; k0 < bs; k0 += 16)
        mma_split(d, &sm.ST[(s0 + bs + 16 * tm) * LDF + s0 + bs + k0], LDF,
                  &sm.Y[(p * bs + k0) * LDY + 8 * tn], LDY, lane);
      float* o0 = &sm.ST[(s0 + bs + 16 * tm + g4) * LDF + s0 + 8 * tn + 2 * t4];
      o0[0] = -d[0];
      o0[1] = -d[1];
      o0[8 * LDF] = -d[2];
      o0[8 * LDF + 1] = -d[3];
    }
    __syncthreads();
  }

  if (a.T_dbg) {
    float* dst = a.T_dbg + chunk_id * CH * CH;
    for (int i = tid; i < CH * CH; i += NTHREADS) dst[i] = sm.ST[(i >> 7) * LDF + (i & 127)];
  }
  if (a.Tb) {
    bf16* dst = a.Tb + chunk_id * CH * CH;
    for (int i = tid; i < CH * CH / 2; i += NTHREADS) {
      const int r = (2 * i) >> 7, cc = (2 * i) & 127;
      *reinterpret_cast<uint32_t*>(dst + 2 * i) =
          pack_bf16(sm.ST[r * LDF + cc], sm.ST[r * LDF + cc + 1]);
    }
  }

  // ---- w = T diag(beta gamma) K ------------------------------------------------
  if (a.W) {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      if (ks <= warp) {  // T is lower triangular
        uint32_t af[4];
        lda_f32_colscaled(af, sm.ST, m0, ks * 16, sm.bg, lane);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t bb[4];
          ldb_kn(bb, sm.K, LDB, ks * 16, np * 16, lane);
          mma16816(acc[2 * np], af, bb[0], bb[1]);
          mma16816(acc[2 * np + 1], af, bb[2], bb[3]);
        }
      }
    }
    store_rows_bf16(a.W + chunk_id * CH * HD, HD, m0, acc, lane);
  }
  // ---- u = T diag(beta) V ------------------------------------------------------
  cp_async_wait<0>();
  __syncthreads();
  if (needU) {
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      if (ks <= warp) {
        uint32_t af[4];
        lda_f32_colscaled(af, sm.ST, m0, ks * 16, sm.beta, lane);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t bb[4];
          ldb_kn(bb, sm.QV, LDB, ks * 16, np * 16, lane);
          mma16816(acc[2 * np], af, bb[0], bb[1]);
          mma16816(acc[2 * np + 1], af, bb[2], bb[3]);
        }
      }
    }
    store_rows_bf16(a.U + chunk_id * CH * HD, HD, m0, acc, lane);
  }
}

}  // namespace

size_t prep_smem_bytes() { return sizeof(PrepSmem); }

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(PrepSmem);
  cudaError_t e = cudaFuncSetAttribute(k_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.NC, a.Hv, a.B);
  k_prep<<<grid, NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
