// gdn_prep.cu -- per-chunk UT/WY preparation of the chunked gated delta rule.
//
// One CTA per (chunk c, key head, batch row b) serves every value head j that
// shares the key head.  For the 128 rows of the chunk (zero-padded past T
// with g = 0, beta = 0):
//   K K^T and Q K^T              tcgen05 products into tensor memory (once per key head)
//   gates  G = chunk-local cumsum of g, gamma = exp(G)               (per value head)
//   S = tril(diag(beta) (K K^T * M), -1),  M_rs = exp(G_r - G_s) for s <= r,
//       the exponent masked before exp so nothing overflows
//   P = (Q K^T) * M, diagonal included                               (for the output)
//   T = (I + S)^-1 by the blockwise doubling ladder
//   w = T diag(beta gamma) K,  u = T diag(beta) V                     tcgen05 products
// The ladder ("Fuse the Gated Delta Net inter-chunk scan into a Pallas TPU
// kernel", section "Changes", triangular inversion kernel): with X the inverse
// of I + S on its diagonal blocks of size b, the inverse on blocks of size 2b
// is X - X S_l X, S_l the lower-left b x b block of each 2b x 2b diagonal
// block.  The 16 x 16 diagonal blocks are inverted exactly in fp32 by forward
// substitution (one warp per block; the ladder's levels b = 1..8 in one exact
// step) and the levels b = 16, 32, 64 run on the tensor cores with two-term
// bf16 operand splitting (hi*hi + hi*lo + lo*hi, fp32 accumulate), keeping T
// at fp32-like accuracy.  At level b the only new block is the lower-left one,
// -X_D S_C X_A, computed as Y = S_C X_A, then -X_D Y.
// w and u take T rounded to bf16 after the column scaling, as tensor-core
// operands; they are bf16 outputs themselves.
#include "gdn_kernels.cuh"
#include "gdn_tc05.cuh"

namespace gdn {

namespace {

constexpr int LDF = HD + 4;  // fp32 row stride of the S/T tile (float4 rows, 16-byte aligned)
constexpr int LDY = 64 + 4;  // fp32 row stride of the ladder scratch
constexpr float LOG2E = 1.4426950408889634f;

struct PrepSmem {
  bf16 Q[CH * HD];   // SW128 [s][d]: Q, then V^T of the current value head ([v][s])
  bf16 K[CH * HD];   // SW128 [s][d]
  bf16 Kt[CH * HD];  // SW128 [d][s]
  bf16 Tp[CH * HD];  // SW128: raw V staging, then T' = T diag(scale) (A operand of w, u)
  float F[CH * LDF];  // S, overwritten in place by T
  float Y[64 * LDY];
  float Gl[CH], beta[CH], gamma[CH], bg[CH];
  uint64_t bar;
  uint32_t tmem;
  int err;
};

// rows [0, rows) of a [128 x 128] bf16 global tile (row stride gstride) into a
// K-major SW128 shared tile; rows past `rows` are zero-filled
__device__ __forceinline__ void load_sw128_async(bf16* s, const bf16* g, long gstride, int rows,
                                                 int tid) {
  unsigned char* sb = reinterpret_cast<unsigned char*>(s);
#pragma unroll
  for (int i = 0; i < (CH * 16) / NTHREADS; ++i) {
    const int idx = tid + i * NTHREADS;
    const int r = idx >> 4, j = idx & 15;
    const bool ok = r < rows;
    cp_async16(sb + tc::sw128_chunk(r, j, CH), g + (ok ? (long)r * gstride + j * 8 : 0), ok);
  }
}

// dst[c][r] = src[r][c] for two [128 x 128] K-major SW128 tiles; one 8 x 8 block per thread
__device__ __forceinline__ void transpose_sw128(const bf16* src, bf16* dst, int tid) {
  const unsigned char* sb = reinterpret_cast<const unsigned char*>(src);
  unsigned char* db = reinterpret_cast<unsigned char*>(dst);
  const int br = tid >> 4, bc = tid & 15;  // source rows 8br.., source columns 8bc..
  uint32_t in[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 u = *reinterpret_cast<const uint4*>(sb + tc::sw128_chunk(8 * br + i, bc, CH));
    in[i][0] = u.x;
    in[i][1] = u.y;
    in[i][2] = u.z;
    in[i][3] = u.w;
  }
  // element (i, c) of the block: half (c & 1) of word in[i][c >> 1]
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t lo = in[2 * p][c >> 1], hi = in[2 * p + 1][c >> 1];
      w[p] = (c & 1) ? __byte_perm(lo, hi, 0x7632) : __byte_perm(lo, hi, 0x5410);
    }
    *reinterpret_cast<uint4*>(db + tc::sw128_chunk(8 * bc + c, br, CH)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

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

// T = (I + S)^-1 in place in F (all threads of the CTA).
__device__ __forceinline__ void ut_inverse(PrepSmem& sm, int warp, int lane) {
  const int g4 = lane >> 2, t4 = lane & 3;
  // (1) exact forward substitution of the 16x16 diagonal block of this warp;
  //     lane j (< 16) carries column j of the block in t[]
  {
    const int base = 16 * warp;
    const int jl = lane & 15;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float* srow = &sm.F[(base + i) * LDF + base];
      float x = (jl == i) ? 1.f : 0.f;
#pragma unroll
      for (int s = 0; s < i; ++s) x -= srow[s] * t[s];
      t[i] = x;
    }
    __syncwarp();
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) sm.F[(base + i) * LDF + base + lane] = t[i];
    }
  }
  __syncthreads();
  // (2) ladder levels b = 16, 32, 64 on the lower-left blocks
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
        mma_split(d, &sm.F[(s0 + bs + 16 * tm) * LDF + s0 + k0], LDF,
                  &sm.F[(s0 + k0) * LDF + s0 + 8 * tn], LDF, lane);
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
        mma_split(d, &sm.F[(s0 + bs + 16 * tm) * LDF + s0 + bs + k0], LDF,
                  &sm.Y[(p * bs + k0) * LDY + 8 * tn], LDY, lane);
      float* o0 = &sm.F[(s0 + bs + 16 * tm + g4) * LDF + s0 + 8 * tn + 2 * t4];
      o0[0] = -d[0];
      o0[1] = -d[1];
      o0[8 * LDF] = -d[2];
      o0[8 * LDF + 1] = -d[3];
    }
    __syncthreads();
  }
}

// T' = T diag(scale) rounded to bf16 into the SW128 tile Tp.
__device__ __forceinline__ void build_tprime(PrepSmem& sm, const float* scale, int tid) {
  unsigned char* tb = reinterpret_cast<unsigned char*>(sm.Tp);
#pragma unroll
  for (int i = 0; i < (CH * 16) / NTHREADS; ++i) {
    const int idx = tid + i * NTHREADS;
    const int r = idx >> 4, j = idx & 15;
    const float4 a = *reinterpret_cast<const float4*>(&sm.F[r * LDF + 8 * j]);
    const float4 b = *reinterpret_cast<const float4*>(&sm.F[r * LDF + 8 * j + 4]);
    const float4 sa = *reinterpret_cast<const float4*>(&scale[8 * j]);
    const float4 sb = *reinterpret_cast<const float4*>(&scale[8 * j + 4]);
    uint4 o;
    o.x = pack_bf16(a.x * sa.x, a.y * sa.y);
    o.y = pack_bf16(a.z * sa.z, a.w * sa.w);
    o.z = pack_bf16(b.x * sb.x, b.y * sb.y);
    o.w = pack_bf16(b.z * sb.z, b.w * sb.w);
    *reinterpret_cast<uint4*>(tb + tc::sw128_chunk(r, j, CH)) = o;
  }
}

// 64 columns (half hh) of this thread's TMEM row -> bf16 in global memory:
// columns 0..31 to dst0, 32..63 to dst1
__device__ __forceinline__ void tmem_row_to_bf16(uint32_t taddr, bf16* dst0, bf16* dst1) {
#pragma unroll
  for (int cb = 0; cb < 64; cb += 32) {
    float v[32];
    tc::ld32(taddr + cb, v);
    bf16* dst = cb ? dst1 : dst0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 o;
      o.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
      o.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
      o.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
      o.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
      *reinterpret_cast<uint4*>(dst + 8 * q) = o;
    }
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) k_prep(PrepArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(base);
  const int c = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = a.Hv / a.Hk;
  const int t0 = c * CH;
  const int L = min(CH, a.T - t0);
  const long tokstride = (long)a.Hk * HD;
  const bf16* kgl = a.k + (((long)b * a.T + t0) * a.Hk + kh) * HD;
  const bf16* qgl = a.q + (((long)b * a.T + t0) * a.Hk + kh) * HD;
  const bool needP = a.P != nullptr;
  const bool needU = a.U != nullptr;
  // TMEM row of this thread in the epilogues: lane quarter of the warp, column half
  const int quarter = warp & 3, hh = warp >> 2;
  const int row = 32 * quarter + lane;
  const long tileP = (long)CH * CH;  // w, u and P tiles: [128][128] row-major
  const int ldP = CH;

  load_sw128_async(sm.K, kgl, tokstride, L, tid);
  if (needP) load_sw128_async(sm.Q, qgl, tokstride, L, tid);
  cp_async_commit();
  if (warp == 0) tc::alloc(&sm.tmem, 512);
  if (tid == 0) {
    tc::mbar_init(&sm.bar, 1);
    tc::mbar_fence_init();
    sm.err = 0;
  }
  cp_async_wait<0>();
  __syncthreads();
  transpose_sw128(sm.K, sm.Kt, tid);
  tc::fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t tlane = tmem + ((uint32_t)(32 * quarter) << 16);
  if (tid == 0) {
    tc::gemm_k128(tmem + 0, smem_u32(sm.K), smem_u32(sm.K), 128, false);
    if (needP) tc::gemm_k128(tmem + 128, smem_u32(sm.Q), smem_u32(sm.K), 128, false);
    tc::commit(&sm.bar);
  }
  uint32_t phase = 0;
  bool ok = true;

  for (int jj = 0; jj < group && ok; ++jj) {
    const int j = kh * group + jj;
    const long bh = (long)b * a.Hv + j;
    const long chunk_id = bh * a.NC + c;
    // V_j (raw rows) into the T' buffer; gates of value head j
    if (needU) {
      load_sw128_async(sm.Tp, a.v + (((long)b * a.T + t0) * a.Hv + j) * HD, (long)a.Hv * HD, L, tid);
    }
    cp_async_commit();
    float gv = 0.f;
    if (tid < CH) {
      const long idx = ((long)b * a.T + t0 + tid) * a.Hv + j;
      gv = tid < L ? a.g[idx] : 0.f;
      sm.beta[tid] = tid < L ? a.beta[idx] : 0.f;
    }
    if (jj == 0) {  // K K^T and Q K^T are done (they read Q, which V^T overwrites)
      ok = tc::mbar_wait(&sm.bar, phase);
      phase ^= 1;
    }
    tc::fence_after();
    __syncthreads();
    if (tid < CH) sm.Gl[tid] = gv;
    __syncthreads();
    if (warp == 0) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = sm.Gl[lane * 4 + i];
      warp_cumsum128(v, lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane * 4 + i;
        const float gm = expf(v[i]);
        sm.Gl[r] = v[i] * LOG2E;
        sm.gamma[r] = gm;
        sm.bg[r] = sm.beta[r] * gm;
      }
    }
    cp_async_wait<0>();
    __syncthreads();
    if (needU) transpose_sw128(sm.Tp, sm.Q, tid);  // V^T: [v][s]

    // ---- S (fp32, into F) and P (bf16, to global) from K K^T and Q K^T -------
    {
      const float Glr = sm.Gl[row], br = sm.beta[row];
      const bool upper = (64 * hh) >= (32 * quarter + 32);  // block entirely above the diagonal
#pragma unroll
      for (int cb = 0; cb < 64; cb += 32) {
        const int c0 = 64 * hh + cb;
        float v[32];
        if (!upper) {
          tc::ld32(tlane + c0, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int s = c0 + i;
            v[i] = (s < row) ? br * v[i] * exp2f(Glr - sm.Gl[s]) : 0.f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(&sm.F[row * LDF + c0 + 4 * q]) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      if (needP) {
        bf16* prow = a.P + chunk_id * tileP + (long)row * ldP + 64 * hh;
#pragma unroll
        for (int cb = 0; cb < 64; cb += 32) {
          const int c0 = 64 * hh + cb;
          float v[32];
          if (!upper) {
            tc::ld32(tlane + 128 + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int s = c0 + i;
              v[i] = (s <= row) ? v[i] * exp2f(Glr - sm.Gl[s]) : 0.f;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
            o.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
            o.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
            o.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
            *reinterpret_cast<uint4*>(prow + cb + 8 * q) = o;
          }
        }
      }
    }
    __syncthreads();
    if (a.S_dbg) {
      float* dst = a.S_dbg + chunk_id * CH * CH;
      for (int i = tid; i < CH * CH; i += NTHREADS) dst[i] = sm.F[(i >> 7) * LDF + (i & 127)];
      __syncthreads();
    }

    // ---- T = (I + S)^-1 -------------------------------------------------------------
    ut_inverse(sm, warp, lane);
    if (a.T_dbg) {
      float* dst = a.T_dbg + chunk_id * CH * CH;
      for (int i = tid; i < CH * CH; i += NTHREADS) dst[i] = sm.F[(i >> 7) * LDF + (i & 127)];
    }
    if (a.Tb) {
      bf16* dst = a.Tb + chunk_id * CH * CH;
      for (int i = tid; i < CH * CH / 2; i += NTHREADS) {
        const int r = (2 * i) >> 7, cc = (2 * i) & 127;
        *reinterpret_cast<uint32_t*>(dst + 2 * i) = pack_bf16(sm.F[r * LDF + cc], sm.F[r * LDF + cc + 1]);
      }
    }
    // ---- w = T diag(beta gamma) K --------------------------------------------------
    if (a.W) {
      build_tprime(sm, sm.bg, tid);
      tc::fence_proxy_async();
      tc::fence_before();
      __syncthreads();
      tc::fence_after();
      if (tid == 0) {
        tc::gemm_k128(tmem + 256, smem_u32(sm.Tp), smem_u32(sm.Kt), 128, false);
        tc::commit(&sm.bar);
      }
      ok = ok && tc::mbar_wait(&sm.bar, phase);
      phase ^= 1;
      tc::fence_after();
      bf16* wrow = a.W + chunk_id * tileP + (long)row * ldP + 64 * hh;
      tmem_row_to_bf16(tlane + 256 + 64 * hh, wrow, wrow + 32);
      tc::fence_before();
      __syncthreads();  // the w product has finished reading T'
      tc::fence_after();
    }
    // ---- u = T diag(beta) V ----------------------------------------------------------
    if (needU) {
      build_tprime(sm, sm.beta, tid);
      tc::fence_proxy_async();
      tc::fence_before();
      __syncthreads();
      tc::fence_after();
      if (tid == 0) {
        tc::gemm_k128(tmem + 384, smem_u32(sm.Tp), smem_u32(sm.Q), 128, false);
        tc::commit(&sm.bar);
      }
      ok = ok && tc::mbar_wait(&sm.bar, phase);
      phase ^= 1;
      tc::fence_after();
      bf16* urow = a.U + chunk_id * CH * HD + (long)row * HD + 64 * hh;
      tmem_row_to_bf16(tlane + 384 + 64 * hh, urow, urow + 32);
    }
    tc::fence_before();
    __syncthreads();  // T', V^T and F are free for the next value head
    tc::fence_after();
  }
  if (!ok && a.status && lane == 0) atomicOr(a.status, 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

}  // namespace

size_t prep_smem_bytes() { return sizeof(PrepSmem) + 1024; }

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  const size_t smem = prep_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.NC, a.Hk, a.B);
  k_prep<<<grid, NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
