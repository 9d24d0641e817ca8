// gdn_walk_bwd.cu -- reverse walk of the state cotangent over the chunks of a segment.
//
// The backward "walks the chunks in reverse" ("Fuse the Gated Delta Net
// inter-chunk scan into a Pallas TPU kernel", section "Changes").  With dh the
// cotangent of the state leaving chunk c, the chunk forward
//     Delta = u - w h,  O = diag(gamma) Q h + P Delta,  h' = gamma_C h + k_g^T Delta
// gives
//     dDelta = P^T dO + k_g dh'                          (= Y below)
//     dh     = gamma_C dh' + Q^T diag(gamma) dO - w^T dDelta,
// an affine map of dh' with matrix A_c^T, so it segments exactly like the
// forward (the transposed maps compose in reverse order).  Each CTA owns a
// 32-column slice of dh (columns are independent) in fp32 registers.
// The chunk tiles stream, in the order they are consumed (K, P, then Q, w),
// through a ring of padded shared buffers, each requested with cp.async
// (one commit group per tile) about a chunk before it is needed; the CTA's dO
// columns are double-buffered.
//
// Modes:
//   WALK (fold = 0): from the cotangent leaving the segment, store for every
//     chunk the bf16 cotangent of the state leaving it and dDelta; segment 0
//     writes dh0 (the cotangent of the initial state).
//   FOLD (fold = 1): push [Abar | Bbar] from [I | 0] backwards through the
//     segment's chunks; the Abar columns take no dO terms.  The result maps
//     the cotangent leaving the segment to the one entering it:
//     dh_in = Abar dh_out + Bbar.
#include "gdn_kernels.cuh"

namespace gdn {

namespace {

constexpr int NSLOT_MAX = 5;

struct WalkBwdSmem {
  bf16 slot[NSLOT_MAX][CH * LDB];  // padded 128 x 128 tiles
  bf16 dO[2][CH * LDS_];
  bf16 dOg[CH * LDS_];
  bf16 X[HD * LDS_];
  bf16 Yn[CH * LDS_];
  float gamma[2][CH];
  float ef[2][CH];
  float gC[2];
};

__device__ __forceinline__ void chunk_gates_b(float (&v)[4], float* gamma, float* ef, float* gC,
                                              int lane) {
  warp_cumsum128(v, lane);
  const float Glast = __shfl_sync(0xffffffffu, v[3], 31);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    gamma[lane * 4 + i] = expf(v[i]);
    ef[lane * 4 + i] = expf(Glast - v[i]);
  }
  if (lane == 0) *gC = expf(Glast);
}

template <bool FOLD>
__global__ void __launch_bounds__(NTHREADS, 1) k_walk_bwd(WalkBwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  WalkBwdSmem& sm = *reinterpret_cast<WalkBwdSmem*>(smem_raw);
  const int slice = blockIdx.x, seg = blockIdx.y, bhi = blockIdx.z;
  const int b = bhi / a.Hv, j = bhi % a.Hv, kh = j / (a.Hv / a.Hk);
  const long bh = bhi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int cbeg = (int)((long)seg * a.NC / a.S), cend = (int)((long)(seg + 1) * a.NC / a.S);
  const bool partA = FOLD && slice < 4;  // Abar columns: no dO terms
  const bool withO = !partA;
  const int TPC = withO ? 4 : 2;  // tiles per chunk: K, P, Q, w  (or K, w)
  const int NSLOT = withO ? 5 : 4;
  const int ntiles = (cend - cbeg) * TPC;
  const int col0 = (slice & 3) * SL;
  const int m0 = warp * 16;
  const int r0 = m0 + g4, r1 = r0 + 8;
  const long tokstride = (long)a.Hk * HD;
  if (cbeg >= cend) return;

  float x[4][4];
  if (FOLD) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = col0 + nt * 8 + 2 * t4 + e;
        x[nt][e] = (partA && r0 == col) ? 1.f : 0.f;
        x[nt][2 + e] = (partA && r1 == col) ? 1.f : 0.f;
      }
  } else {
    const float* hs = a.hstart ? a.hstart + bh * a.hstart_bh_stride + seg * a.hstart_seg_stride : nullptr;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = col0 + nt * 8 + 2 * t4;
      float2 x0 = make_float2(0.f, 0.f), x1 = x0;
      if (hs) {
        x0 = *reinterpret_cast<const float2*>(hs + r0 * HD + col);
        x1 = *reinterpret_cast<const float2*>(hs + r1 * HD + col);
      }
      x[nt][0] = x0.x;
      x[nt][1] = x0.y;
      x[nt][2] = x1.x;
      x[nt][3] = x1.y;
    }
  }

  auto rows_of = [&](int c) { return min(CH, a.T - c * CH); };
  auto tok = [&](int c) { return (long)b * a.T + (long)c * CH; };
  // request tile i of the reverse sequence (every thread; one commit group per tile)
  auto issue = [&](int i) {
    if (i < ntiles) {
      const int ci = i / TPC, t = i % TPC;
      const int c = cend - 1 - ci;
      const long cid = bh * a.NC + c;
      bf16* dst = sm.slot[i % NSLOT];
      const int kind = withO ? t : (t == 0 ? 0 : 3);  // 0 K, 1 P, 2 Q, 3 w
      if (kind == 0) {
        tile_load_async(dst, a.k + (tok(c) * a.Hk + kh) * HD, tokstride, rows_of(c), tid);
        if (withO)
          slice_load_async(sm.dO[ci & 1], a.dO + (tok(c) * a.Hv + j) * HD + col0, (long)a.Hv * HD,
                           rows_of(c), tid);
      } else if (kind == 1) {
        tile_load_async(dst, a.P + cid * CH * CH, CH, CH, tid);
      } else if (kind == 2) {
        tile_load_async(dst, a.q + (tok(c) * a.Hk + kh) * HD, tokstride, rows_of(c), tid);
      } else {
        tile_load_async(dst, a.W + cid * CH * HD, HD, CH, tid);
      }
    }
    cp_async_commit();
  };
  auto load_g = [&](int c, float (&v)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      v[i] = (c >= cbeg && r < rows_of(c)) ? a.g[(tok(c) + r) * a.Hv + j] : 0.f;
    }
  };

  for (int i = 0; i < NSLOT; ++i) issue(i);
  float gnext[4];
  if (warp == 0) {
    float v[4];
    load_g(cend - 1, v);
    chunk_gates_b(v, sm.gamma[(cend - 1) & 1], sm.ef[(cend - 1) & 1], &sm.gC[(cend - 1) & 1], lane);
    load_g(cend - 2, gnext);
  }

  for (int c = cend - 1; c >= cbeg; --c) {
    const int ci = cend - 1 - c;
    const int par = c & 1;
    const int tk = ci * TPC;  // index of this chunk's K tile
    const bf16* sK = sm.slot[tk % NSLOT];
    const bf16* sP = sm.slot[(tk + 1) % NSLOT];
    const bf16* sQ = sm.slot[(tk + 2) % NSLOT];
    const bf16* sW = sm.slot[(tk + (withO ? 3 : 1)) % NSLOT];
    const bf16* sdO = sm.dO[ci & 1];
    cp_async_wait_n(3);  // K, dO (and P): NSLOT + tk groups committed
    // bf16 image of dh' (B operand), its export, and gamma * dO
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(sm.X + r0 * LDS_ + col) = pack_bf16(x[nt][0], x[nt][1]);
      *reinterpret_cast<uint32_t*>(sm.X + r1 * LDS_ + col) = pack_bf16(x[nt][2], x[nt][3]);
    }
    if (!FOLD) {
      bf16* st = a.dstates + ((bh * a.NC + c) * HD) * HD + col0;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = nt * 8 + 2 * t4;
        *reinterpret_cast<uint32_t*>(st + (long)r0 * HD + col) = pack_bf16(x[nt][0], x[nt][1]);
        *reinterpret_cast<uint32_t*>(st + (long)r1 * HD + col) = pack_bf16(x[nt][2], x[nt][3]);
      }
    }
    __syncthreads();  // dO landed for every thread's copy, gates and the dh' image visible
    if (withO) {
      // 128 rows x 32 cols: 2 rows of 8 columns per thread
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int idx = tid + i * NTHREADS;
        const int r = idx >> 2, c8 = (idx & 3) << 3;
        const float gm = sm.gamma[par][r];
        uint4 raw = *reinterpret_cast<const uint4*>(sdO + r * LDS_ + c8);
        uint32_t* w = reinterpret_cast<uint32_t*>(&raw);
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          float2 f = unpack_bf16(w[q2]);
          w[q2] = pack_bf16(gm * f.x, gm * f.y);
        }
        *reinterpret_cast<uint4*>(sm.dOg + r * LDS_ + c8) = raw;
      }
    }

    // ---- Y = dDelta = diag(ef) K dh' + P^T dO ---------------------------------
    float y[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i][0] = y[i][1] = y[i][2] = y[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t af[4], bb[4];
      lda_rm(af, sK, LDB, m0, ks * 16, lane);
      ldb_kn(bb, sm.X, LDS_, ks * 16, 0, lane);
      mma16816(y[0], af, bb[0], bb[1]);
      mma16816(y[1], af, bb[2], bb[3]);
      ldb_kn(bb, sm.X, LDS_, ks * 16, 16, lane);
      mma16816(y[2], af, bb[0], bb[1]);
      mma16816(y[3], af, bb[2], bb[3]);
    }
    {
      const float e0 = sm.ef[par][r0], e1 = sm.ef[par][r1];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        y[nt][0] *= e0;
        y[nt][1] *= e0;
        y[nt][2] *= e1;
        y[nt][3] *= e1;
      }
    }
    if (withO) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (ks >= warp) {  // P^T is upper triangular
          uint32_t af[4], bb[4];
          lda_tr(af, sP, LDB, m0, ks * 16, lane);
          ldb_kn(bb, sdO, LDS_, ks * 16, 0, lane);
          mma16816(y[0], af, bb[0], bb[1]);
          mma16816(y[1], af, bb[2], bb[3]);
          ldb_kn(bb, sdO, LDS_, ks * 16, 16, lane);
          mma16816(y[2], af, bb[0], bb[1]);
          mma16816(y[3], af, bb[2], bb[3]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(sm.Yn + r0 * LDS_ + col) = pack_bf16(-y[nt][0], -y[nt][1]);
      *reinterpret_cast<uint32_t*>(sm.Yn + r1 * LDS_ + col) = pack_bf16(-y[nt][2], -y[nt][3]);
      if (!FOLD) {
        bf16* dd = a.ddelta + ((bh * a.NC + c) * CH) * HD + col0 + col;
        *reinterpret_cast<uint32_t*>(dd + (long)r0 * HD) = pack_bf16(y[nt][0], y[nt][1]);
        *reinterpret_cast<uint32_t*>(dd + (long)r1 * HD) = pack_bf16(y[nt][2], y[nt][3]);
      }
    }
    // NSLOT + tk groups committed; Q and w are tiles tk+2, tk+3 (or w = tk+1)
    cp_async_wait_n(withO ? 1 : 2);
    __syncthreads();  // K, P consumed; Yn, dOg complete; Q, w visible
    issue(tk + NSLOT);
    if (withO) issue(tk + 1 + NSLOT);

    // ---- dh = gamma_C dh' + Q^T (gamma dO) + W^T (-Y) -----------------------------
    {
      const float gC = sm.gC[par];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[nt][e] *= gC;
      if (withO) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t af[4], bb[4];
          lda_tr(af, sQ, LDB, m0, ks * 16, lane);
          ldb_kn(bb, sm.dOg, LDS_, ks * 16, 0, lane);
          mma16816(x[0], af, bb[0], bb[1]);
          mma16816(x[1], af, bb[2], bb[3]);
          ldb_kn(bb, sm.dOg, LDS_, ks * 16, 16, lane);
          mma16816(x[2], af, bb[0], bb[1]);
          mma16816(x[3], af, bb[2], bb[3]);
        }
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4], bb[4];
        lda_tr(af, sW, LDB, m0, ks * 16, lane);
        ldb_kn(bb, sm.Yn, LDS_, ks * 16, 0, lane);
        mma16816(x[0], af, bb[0], bb[1]);
        mma16816(x[1], af, bb[2], bb[3]);
        ldb_kn(bb, sm.Yn, LDS_, ks * 16, 16, lane);
        mma16816(x[2], af, bb[0], bb[1]);
        mma16816(x[3], af, bb[2], bb[3]);
      }
    }
    __syncthreads();  // Q, w, dOg, X, Yn consumed
    if (withO) {
      issue(tk + 2 + NSLOT);
      issue(tk + 3 + NSLOT);
    } else {
      issue(tk + 1 + NSLOT);
    }
    if (warp == 0 && c - 1 >= cbeg) {
      chunk_gates_b(gnext, sm.gamma[par ^ 1], sm.ef[par ^ 1], &sm.gC[par ^ 1], lane);
      load_g(c - 2, gnext);
    }
  }
  cp_async_wait<0>();

  if (FOLD) {
    float* dst = (partA ? a.pairA : a.pairB) + (bh * a.S + seg) * HD * HD + col0;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(dst + r0 * HD + col) = make_float2(x[nt][0], x[nt][1]);
      *reinterpret_cast<float2*>(dst + r1 * HD + col) = make_float2(x[nt][2], x[nt][3]);
    }
  } else if (a.dh0 && seg == 0) {
    float* dst = a.dh0 + bh * HD * HD + col0;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(dst + r0 * HD + col) = make_float2(x[nt][0], x[nt][1]);
      *reinterpret_cast<float2*>(dst + r1 * HD + col) = make_float2(x[nt][2], x[nt][3]);
    }
  }
}

}  // namespace

size_t walk_bwd_smem_bytes(int) { return sizeof(WalkBwdSmem); }

cudaError_t launch_walk_bwd(const WalkBwdArgs& a, int fold, cudaStream_t s) {
  const size_t smem = sizeof(WalkBwdSmem);
  cudaError_t e;
  if (fold) {
    e = cudaFuncSetAttribute(k_walk_bwd<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_walk_bwd<true><<<dim3(8, a.S, a.B * a.Hv), NTHREADS, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(k_walk_bwd<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_walk_bwd<false><<<dim3(HD / SL, a.S, a.B * a.Hv), NTHREADS, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
