// gdn_walk_fwd.cu -- sequential forward walk over the chunks of a segment.
//
// Inter-chunk step ("GatedDeltaNet does not support ici_context_parallelism",
// section "The recurrence is affine, so it can be parallelized"):
//     Delta = u - w h,     h' = exp(g_last) h + k_g^T Delta,
// with k_g = diag(exp(G_last - G)) K, and the masked intra-chunk output
//     O = diag(gamma) Q h + P Delta,      P = (Q K^T) * decay (diagonal included).
//
// The state h (128 x 128 fp32) never leaves the SM while a segment is walked:
// each CTA owns a 32-column slice of h (the matrices of the step act on h from
// the left only, so columns evolve independently), kept in mma accumulator
// registers; its bf16 image in shared memory is the B operand of the next
// chunk's w h and Q h.
//
// The chunk tiles stream through a ring of NSLOT padded shared buffers in the
// order they are consumed (w, K, then Q, P when the output is produced).  Tile
// i goes to slot i % NSLOT and is requested as soon as tile i - NSLOT has been
// consumed, so every tile is in flight for about a chunk before it is needed.
// A tile is requested with cp.async (16 bytes per thread and copy, one commit
// group per tile, so "tile i has landed" is a group count); u (the CTA's own
// 32 columns) is double-buffered by chunk parity and travels with its chunk's
// w tile.
//
// Modes:
//   RECUR (fold = 0): walk from the segment's entering state, write O (if o
//     is given), and optionally the bf16 entering state and Delta of every
//     chunk (backward recomputation) and the final state (last segment).
//   FOLD  (fold = 1): pass 1 of the two-pass segment scan ("Shard the
//     GatedDeltaNet sequence under ici_context_parallelism", description):
//     push the augmented state [A | B] through the segment's chunks starting
//     from [I | 0]; the A columns take no u term.  CTAs 0-3 hold A's column
//     slices, 4-7 hold B's.
#include "gdn_kernels.cuh"

namespace gdn {

namespace {

constexpr int NSLOT_MAX = 5;

struct WalkFwdSmem {
  bf16 slot[NSLOT_MAX][CH * LDB];  // padded 128 x 128 tiles
  bf16 U[2][CH * LDS_];
  bf16 H[HD * LDS_];
  bf16 D[CH * LDS_];
  bf16 Dg[CH * LDS_];
  float gamma[2][CH];
  float ef[2][CH];
  float gC[2];
};

// Gates of one chunk from the 128 log-gates held 4 per lane by warp 0.
__device__ __forceinline__ void chunk_gates(float (&v)[4], float* gamma, float* ef, float* gC,
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
__global__ void __launch_bounds__(NTHREADS, 1) k_walk_fwd(WalkFwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  WalkFwdSmem& sm = *reinterpret_cast<WalkFwdSmem*>(smem_raw);
  const int slice = blockIdx.x, seg = blockIdx.y, bhi = blockIdx.z;
  const int b = bhi / a.Hv, j = bhi % a.Hv, kh = j / (a.Hv / a.Hk);
  const long bh = bhi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int cbeg = (int)((long)seg * a.NC / a.S), cend = (int)((long)(seg + 1) * a.NC / a.S);
  const bool partA = FOLD && slice < 4;  // A columns: no u term
  const bool withO = !FOLD && a.o != nullptr;
  const int TPC = withO ? 4 : 2;                 // tiles per chunk: w, K (, Q, P)
  const int NSLOT = withO ? 5 : 4;
  const int ntiles = (cend - cbeg) * TPC;
  const int col0 = (slice & 3) * SL;
  const int m0 = warp * 16;
  const int r0 = m0 + g4, r1 = r0 + 8;
  const long tokstride = (long)a.Hk * HD;
  if (cbeg >= cend) return;

  auto rows_of = [&](int c) { return min(CH, a.T - c * CH); };
  // request tile i (every thread; always commits exactly one cp.async group)
  auto issue = [&](int i) {
    if (i < ntiles) {
      const int c = cbeg + i / TPC, t = i % TPC;
      const long cid = bh * a.NC + c;
      bf16* dst = sm.slot[i % NSLOT];
      if (t == 0) {
        tile_load_async(dst, a.W + cid * CH * HD, HD, CH, tid);
        if (!partA) slice_load_async(sm.U[c & 1], a.U + cid * CH * HD + col0, HD, CH, tid);
      } else if (t == 1) {
        tile_load_async(dst, a.k + (((long)b * a.T + (long)c * CH) * a.Hk + kh) * HD, tokstride,
                        rows_of(c), tid);
      } else if (t == 2) {
        tile_load_async(dst, a.q + (((long)b * a.T + (long)c * CH) * a.Hk + kh) * HD, tokstride,
                        rows_of(c), tid);
      } else {
        tile_load_async(dst, a.P + cid * CH * CH, CH, CH, tid);
      }
    }
    cp_async_commit();
  };
  auto load_g = [&](int c, float (&v)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      v[i] = (c < cend && r < rows_of(c)) ? a.g[((long)b * a.T + (long)c * CH + r) * a.Hv + j] : 0.f;
    }
  };

  // state slice: rows r0, r1 of h; columns col0 + 8 nt + 2 t4 + {0,1}
  float h[4][4];
  if (FOLD) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = col0 + nt * 8 + 2 * t4 + e;
        h[nt][e] = (partA && r0 == col) ? 1.f : 0.f;
        h[nt][2 + e] = (partA && r1 == col) ? 1.f : 0.f;
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
      h[nt][0] = x0.x;
      h[nt][1] = x0.y;
      h[nt][2] = x1.x;
      h[nt][3] = x1.y;
    }
  }

  for (int i = 0; i < NSLOT; ++i) issue(i);
  float gnext[4];
  if (warp == 0) {
    float v[4];
    load_g(cbeg, v);
    chunk_gates(v, sm.gamma[cbeg & 1], sm.ef[cbeg & 1], &sm.gC[cbeg & 1], lane);
    load_g(cbeg + 1, gnext);
  }

  for (int c = cbeg; c < cend; ++c) {
    const int ci = c - cbeg;
    const int par = c & 1;
    const int tw = ci * TPC;  // index of this chunk's w tile
    const bf16* sW = sm.slot[tw % NSLOT];
    const bf16* sK = sm.slot[(tw + 1) % NSLOT];
    const bf16* sU = sm.U[c & 1];
    // tiles <= tw + 1 (w, u, K) are needed; NSLOT + tw groups have been committed
    cp_async_wait_n(NSLOT - 2);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {  // bf16 image of the entering state
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(sm.H + r0 * LDS_ + col) = pack_bf16(h[nt][0], h[nt][1]);
      *reinterpret_cast<uint32_t*>(sm.H + r1 * LDS_ + col) = pack_bf16(h[nt][2], h[nt][3]);
    }
    if (!FOLD && a.states) {
      bf16* st = a.states + ((bh * a.NC + c) * HD) * HD + col0;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = nt * 8 + 2 * t4;
        *reinterpret_cast<uint32_t*>(st + (long)r0 * HD + col) = pack_bf16(h[nt][0], h[nt][1]);
        *reinterpret_cast<uint32_t*>(st + (long)r1 * HD + col) = pack_bf16(h[nt][2], h[nt][3]);
      }
    }
    __syncthreads();  // w, K, u of chunk c, the state image and the gates are ready

    // ---- X = w h;  Delta = u - X -----------------------------------------------
    float x[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) x[q][0] = x[q][1] = x[q][2] = x[q][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t af[4], bb[4];
      lda_rm(af, sW, LDB, m0, ks * 16, lane);
      ldb_kn(bb, sm.H, LDS_, ks * 16, 0, lane);
      mma16816(x[0], af, bb[0], bb[1]);
      mma16816(x[1], af, bb[2], bb[3]);
      ldb_kn(bb, sm.H, LDS_, ks * 16, 16, lane);
      mma16816(x[2], af, bb[0], bb[1]);
      mma16816(x[3], af, bb[2], bb[3]);
    }
    {
      const float e0 = sm.ef[par][r0], e1 = sm.ef[par][r1];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = nt * 8 + 2 * t4;
        float2 u0 = make_float2(0.f, 0.f), u1 = u0;
        if (!partA) {
          u0 = unpack_bf16(*reinterpret_cast<const uint32_t*>(sU + r0 * LDS_ + col));
          u1 = unpack_bf16(*reinterpret_cast<const uint32_t*>(sU + r1 * LDS_ + col));
        }
        const float d00 = u0.x - x[nt][0], d01 = u0.y - x[nt][1];
        const float d10 = u1.x - x[nt][2], d11 = u1.y - x[nt][3];
        if (withO) {
          *reinterpret_cast<uint32_t*>(sm.D + r0 * LDS_ + col) = pack_bf16(d00, d01);
          *reinterpret_cast<uint32_t*>(sm.D + r1 * LDS_ + col) = pack_bf16(d10, d11);
        }
        if (!FOLD && a.delta) {
          bf16* dd = a.delta + ((bh * a.NC + c) * CH) * HD + col0 + col;
          *reinterpret_cast<uint32_t*>(dd + (long)r0 * HD) = pack_bf16(d00, d01);
          *reinterpret_cast<uint32_t*>(dd + (long)r1 * HD) = pack_bf16(d10, d11);
        }
        *reinterpret_cast<uint32_t*>(sm.Dg + r0 * LDS_ + col) = pack_bf16(e0 * d00, e0 * d01);
        *reinterpret_cast<uint32_t*>(sm.Dg + r1 * LDS_ + col) = pack_bf16(e1 * d10, e1 * d11);
      }
    }
    __syncthreads();  // w and u consumed; D, Dg complete
    issue(tw + NSLOT);

    // ---- h' = exp(g_last) h + K^T (ef * Delta) ---------------------------------
    {
      const float gC = sm.gC[par];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) h[nt][e] *= gC;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4], bb[4];
        lda_tr(af, sK, LDB, m0, ks * 16, lane);
        ldb_kn(bb, sm.Dg, LDS_, ks * 16, 0, lane);
        mma16816(h[0], af, bb[0], bb[1]);
        mma16816(h[1], af, bb[2], bb[3]);
        ldb_kn(bb, sm.Dg, LDS_, ks * 16, 16, lane);
        mma16816(h[2], af, bb[0], bb[1]);
        mma16816(h[3], af, bb[2], bb[3]);
      }
    }

    if (withO) {
      const bf16* sQ = sm.slot[(tw + 2) % NSLOT];
      const bf16* sP = sm.slot[(tw + 3) % NSLOT];
      cp_async_wait_n(NSLOT - 3);  // Q, P (tiles tw+2, tw+3); NSLOT + tw + 1 committed
      __syncthreads();             // K consumed
      issue(tw + 1 + NSLOT);
      float o[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q][0] = o[q][1] = o[q][2] = o[q][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4], bb[4];
        lda_rm(af, sQ, LDB, m0, ks * 16, lane);
        ldb_kn(bb, sm.H, LDS_, ks * 16, 0, lane);
        mma16816(o[0], af, bb[0], bb[1]);
        mma16816(o[1], af, bb[2], bb[3]);
        ldb_kn(bb, sm.H, LDS_, ks * 16, 16, lane);
        mma16816(o[2], af, bb[0], bb[1]);
        mma16816(o[3], af, bb[2], bb[3]);
      }
      const float gm0 = sm.gamma[par][r0], gm1 = sm.gamma[par][r1];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        o[nt][0] *= gm0;
        o[nt][1] *= gm0;
        o[nt][2] *= gm1;
        o[nt][3] *= gm1;
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (ks <= warp) {  // P is lower triangular
          uint32_t af[4], bb[4];
          lda_rm(af, sP, LDB, m0, ks * 16, lane);
          ldb_kn(bb, sm.D, LDS_, ks * 16, 0, lane);
          mma16816(o[0], af, bb[0], bb[1]);
          mma16816(o[1], af, bb[2], bb[3]);
          ldb_kn(bb, sm.D, LDS_, ks * 16, 16, lane);
          mma16816(o[2], af, bb[0], bb[1]);
          mma16816(o[3], af, bb[2], bb[3]);
        }
      }
      const int L = rows_of(c);
      bf16* ob = a.o + (((long)b * a.T + (long)c * CH) * a.Hv + j) * HD + col0;
      const long os = (long)a.Hv * HD;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = nt * 8 + 2 * t4;
        if (r0 < L) *reinterpret_cast<uint32_t*>(ob + r0 * os + col) = pack_bf16(o[nt][0], o[nt][1]);
        if (r1 < L) *reinterpret_cast<uint32_t*>(ob + r1 * os + col) = pack_bf16(o[nt][2], o[nt][3]);
      }
      __syncthreads();  // Q, P, D and the state image consumed
      issue(tw + 2 + NSLOT);
      issue(tw + 3 + NSLOT);
    } else {
      __syncthreads();  // K, Dg and the state image consumed
      issue(tw + 1 + NSLOT);
    }
    if (warp == 0 && c + 1 < cend) {
      chunk_gates(gnext, sm.gamma[par ^ 1], sm.ef[par ^ 1], &sm.gC[par ^ 1], lane);
      load_g(c + 2, gnext);
    }
  }
  cp_async_wait<0>();

  if (FOLD) {
    float* dst = (partA ? a.pairA : a.pairB) + (bh * a.S + seg) * HD * HD + col0;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(dst + r0 * HD + col) = make_float2(h[nt][0], h[nt][1]);
      *reinterpret_cast<float2*>(dst + r1 * HD + col) = make_float2(h[nt][2], h[nt][3]);
    }
  } else if (a.hT && seg == a.S - 1) {
    float* dst = a.hT + bh * HD * HD + col0;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = nt * 8 + 2 * t4;
      *reinterpret_cast<float2*>(dst + r0 * HD + col) = make_float2(h[nt][0], h[nt][1]);
      *reinterpret_cast<float2*>(dst + r1 * HD + col) = make_float2(h[nt][2], h[nt][3]);
    }
  }
}

template <bool FOLD>
cudaError_t launch_one(const WalkFwdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(WalkFwdSmem);
  cudaError_t e = cudaFuncSetAttribute(k_walk_fwd<FOLD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_walk_fwd<FOLD><<<dim3(FOLD ? 8 : HD / SL, a.S, a.B * a.Hv), NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t walk_fwd_smem_bytes(int) { return sizeof(WalkFwdSmem); }

cudaError_t launch_walk_fwd(const WalkFwdArgs& a, int fold, cudaStream_t s) {
  return fold ? launch_one<true>(a, s) : launch_one<false>(a, s);
}

}  // namespace gdn
