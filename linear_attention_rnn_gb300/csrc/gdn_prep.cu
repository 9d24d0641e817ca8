// gdn_prep.cu -- per-chunk UT/WY preparation of the chunked gated delta rule.
//
// Persistent CTAs, one per SM, each take a contiguous range of units (batch
// row b, chunk c, key head, value head j), value heads fastest, so a CTA
// serves the value heads of one (chunk, key head) in a row: it loads K and Q
// and forms K K^T and Q K^T once for them.  (The range balances the work to
// within one unit per SM; a grid of one CTA per (chunk, key head) ran in
// ceil(units / 2 / SMs) rounds of two heads.)  For the 128 rows of the chunk
// (zero-padded past T with g = 0, beta = 0):
//   K K^T and Q K^T              tcgen05 products into tensor memory (once per key head)
//   gates  G = chunk-local cumsum of g, gamma = exp(G)               (per value head)
//   S = tril(diag(beta) (K K^T * M), -1),  M_rs = exp(G_r - G_s) for s <= r,
//       the exponent masked before exp so nothing overflows
//   P = (Q K^T) * M, diagonal included (same exponentials as S)      (for the output)
//   T = (I + S)^-1 by the blockwise doubling ladder
//   u = T' V and w = T'' K with T' = T diag(beta), T'' = T diag(beta gamma)
//                                                                    tcgen05 products
// The ladder ("Fuse the Gated Delta Net inter-chunk scan into a Pallas TPU
// kernel", section "Changes", triangular inversion kernel): with X the inverse
// of I + S on its diagonal blocks of size b, the inverse on blocks of size 2b
// is X - X S_l X, S_l the lower-left b x b block of each 2b x 2b diagonal
// block.  The 16 x 16 diagonal blocks are inverted exactly in fp32 by forward
// substitution (the ladder's levels b = 1..8 in one exact step) and the levels
// b = 16, 32, 64 run on the tensor cores.
//
// Precision: S and T are held as pairs of bf16 tiles (x = hi + lo, hi =
// bf16(x), lo = bf16(x - hi): about 16 significant bits), so every ladder
// operand is a plain ldmatrix load; a product is hi*hi + hi*lo + lo*hi with
// fp32 accumulation.  The zero blocks of the triangular factors are skipped.
// T' and T'' are rounded to bf16 as tensor-core operands; w and u are bf16
// outputs themselves.
//
// 64-token chunks (c64): a 128-row tile holds two chunks.  G restarts at row
// 64, S and P keep only their two 64 x 64 diagonal blocks, and the ladder stops
// after level 32, so T, T', T'' are block diagonal and w, u, P of each chunk
// are its own; everything else runs as for 128-token chunks.
//
// Operands arrive by TMA in the 128-byte-swizzled layout: K and Q serve
// K K^T and Q K^T as K-major operands, and K and V serve w and u as MN-major
// B operands as loaded, so nothing is transposed or rescaled in shared memory.  V of the
// next value head is requested while the current one is processed (the Q
// buffer takes the odd heads once Q K^T has completed).
#include "gdn_kernels.cuh"
#include "gdn_tc05.cuh"
#include "gdn_tmap.cuh"

namespace gdn {

namespace {

constexpr uint32_t TILE = CH * HD * 2;  // 32 KiB bf16 tile
constexpr int PT = 512, PW = PT / 32;  // 16 warps: an epilogue thread owns 32 columns of its row
constexpr float LOG2E = 1.4426950408889634f;

struct PrepSmem {
  unsigned char A[3][TILE];  // SW128 [s][d] tiles: K of the key head and V of two value heads,
                             // the roles rotating from one key-head group to the next
  unsigned char Kg[TILE];  // SW128: P staging; T'' = T diag(beta gamma) [r][s]; w staging
  unsigned char Tp[TILE];  // SW128 [r][s]: T diag(beta); during the inverse its scratch
  bf16 Fh[CH * CH];        // S, overwritten in place by T: high parts (XOR-swizzled rows);
                           // at a group's start, its Q (SW128) until Q K^T has read it
  bf16 Fl[CH * CH];        // low parts
  // gates of a value head; the next value head's are built while the current one's
  // products run (its own are last read by the T' / T'' build, before the products)
  float Gl[CH], beta[CH];
  float etab[CH];  // exp2(Gl[c0] - Gl[s]) for the 16-column block c0 of column s
  uint64_t barKQ, barV[2], barM;
  uint32_t tmem;
};
// scratch of the inverse inside Tp
constexpr uint32_t Y_HI = 0, Y_LO = 8192, SD = 16384;  // Y: [64][64] bf16 pair; Sd: [8][16][16] fp32

struct PrepMaps {
  CUtensorMap q, k, v;  // loads: [B, T, H, 128] activations
  CUtensorMap W, U, P;  // stores: [BH * NC * 128, 128] workspace rows
};

// [rows][64] bf16 tile with 128-byte rows, 16-byte chunk j of row r at j ^ (r & 7)
__device__ __forceinline__ bf16* swz64(bf16* base, int r, int j) {
  return base + r * 64 + ((j ^ (r & 7)) << 3);
}

__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  split_bf16(x0, x1, hi, lo);
}
// eight fp32 values -> hi and lo 16-byte chunks
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
  split2(v[0], v[1], hi.x, lo.x);
  split2(v[2], v[3], hi.y, lo.y);
  split2(v[4], v[5], hi.z, lo.z);
  split2(v[6], v[7], hi.w, lo.w);
}
__device__ __forceinline__ void join8(const uint4& hi, const uint4& lo, float* v) {
  const uint32_t h[4] = {hi.x, hi.y, hi.z, hi.w}, l[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = unpack_bf16(h[i]), b = unpack_bf16(l[i]);
    v[2 * i] = a.x + b.x;
    v[2 * i + 1] = a.y + b.y;
  }
}

// d += A B for a 16 x 16 A and two 8-column B tiles, each operand a hi + lo pair
__device__ __forceinline__ void mma_pair(float (&d0)[4], float (&d1)[4], const uint32_t (&ah)[4],
                                         const uint32_t (&al)[4], const uint32_t (&bh)[4],
                                         const uint32_t (&bl)[4]) {
  mma16816(d0, ah, bh[0], bh[1]);
  mma16816(d0, ah, bl[0], bl[1]);
  mma16816(d0, al, bh[0], bh[1]);
  mma16816(d1, ah, bh[2], bh[3]);
  mma16816(d1, ah, bl[2], bl[3]);
  mma16816(d1, al, bh[2], bh[3]);
}

// B fragments (k0..k0+15, n0..n0+15) of a row-major [k][n] [64 x 64] tile
__device__ __forceinline__ void ldb_kn_64(uint32_t (&b)[4], bf16* base, int k0, int n0, int lane) {
  ldsm_x4_t(b, swz64(base, k0 + (lane & 15), (n0 >> 3) + (lane >> 4)));
}

// Columns 32 cq .. 32 cq + 31 of this thread's TMEM row, as bf16, into row
// `row` of a K-major SW128 [128 x 128] staging tile (the layout a tiled TMA
// store with 64-column boxes reads).
__device__ __forceinline__ void tmem_row_to_tile(uint32_t taddr, unsigned char* tile, int row, int cq) {
  float v[32];
  tc::ld32(taddr, v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 o;
    o.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
    o.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    o.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    o.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(tile + tc::sw128_chunk(row, 4 * cq + q, CH)) = o;
  }
}

// element (r, c) of a [128 x 128] XOR-swizzled bf16 tile
__device__ __forceinline__ bf16* fel(bf16* base, int r, int c) { return swz(base, r, c >> 3) + (c & 7); }

// the two halves of a 16 x 16 accumulator pair (rows r, r + 8; columns
// 2t4.. of n-tile h) -> hi/lo 32-bit words at element pointers given per row
__device__ __forceinline__ void store_split(bf16* hi0, bf16* lo0, bf16* hi1, bf16* lo1,
                                            const float (&d)[4], float sign) {
  uint32_t h, l;
  split2(sign * d[0], sign * d[1], h, l);
  *reinterpret_cast<uint32_t*>(hi0) = h;
  *reinterpret_cast<uint32_t*>(lo0) = l;
  split2(sign * d[2], sign * d[3], h, l);
  *reinterpret_cast<uint32_t*>(hi1) = h;
  *reinterpret_cast<uint32_t*>(lo1) = l;
}

// T = (I + S)^-1 in place in (Fh, Fl); the fp32 diagonal 16 x 16 blocks of S
// are in the Sd scratch.  All threads of the CTA.  The ladder's levels stop
// below `lim` (64: the inverse of each 64 x 64 diagonal block, for S with no
// entries outside them).
template <int LIM>
__device__ __forceinline__ void ut_inverse(PrepSmem& sm, int warp, int lane) {
  bf16* Yh = reinterpret_cast<bf16*>(sm.Tp + Y_HI);
  bf16* Yl = reinterpret_cast<bf16*>(sm.Tp + Y_LO);
  const float* Sd = reinterpret_cast<const float*>(sm.Tp + SD);
  const int g4 = lane >> 2, t4 = lane & 3;
  // (1) exact forward substitution of diagonal block `warp` (warps 0-7): lane
  //     j (mod 16) carries column j; lanes 0-15 store the high parts, 16-31 the low parts
  if (warp < CH / 16) {
    const float* blk = Sd + warp * 256;
    const int jl = lane & 15;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float x = (jl == i) ? 1.f : 0.f;
#pragma unroll
      for (int s = 0; s < i; ++s) x -= blk[i * 16 + s] * t[s];
      t[i] = x;
    }
    bf16* F = lane < 16 ? sm.Fh : sm.Fl;
    const int c = 16 * warp + jl;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const bf16 hb = __float2bfloat16_rn(t[i]);
      *fel(F, 16 * warp + i, c) = lane < 16 ? hb : __float2bfloat16_rn(t[i] - __bfloat162float(hb));
    }
  }
  __syncthreads();
  // (2) levels b = 16, 32, 64: for every 2b block pair p (rows s0 = 2bp..),
  //     Y = S_C X_A, then T_C = -X_D Y, in 16 x 16 output tiles
  for (int bs = 16; bs < LIM; bs *= 2) {
    const int nb = bs >> 4, per = nb * nb;
    const int ntiles = (CH / (2 * bs)) * per;
    // (at most 16 tiles per phase: one per warp)
    for (int t = warp; t < ntiles; t += PW) {
      const int p = t / per, tm = (t % per) / nb, tn = t % nb;
      const int s0 = 2 * bs * p;
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kb = tn; kb < nb; ++kb) {  // X_A is lower triangular
        uint32_t ah[4], al[4], bh[4], bl[4];
        lda_rm_s(ah, sm.Fh, s0 + bs + 16 * tm, s0 + 16 * kb, lane);
        lda_rm_s(al, sm.Fl, s0 + bs + 16 * tm, s0 + 16 * kb, lane);
        ldb_kn_s(bh, sm.Fh, s0 + 16 * kb, s0 + 16 * tn, lane);
        ldb_kn_s(bl, sm.Fl, s0 + 16 * kb, s0 + 16 * tn, lane);
        mma_pair(d0, d1, ah, al, bh, bl);
      }
      const int yr = p * bs + 16 * tm + g4;
      store_split(swz64(Yh, yr, 2 * tn) + 2 * t4, swz64(Yl, yr, 2 * tn) + 2 * t4,
                  swz64(Yh, yr + 8, 2 * tn) + 2 * t4, swz64(Yl, yr + 8, 2 * tn) + 2 * t4, d0, 1.f);
      store_split(swz64(Yh, yr, 2 * tn + 1) + 2 * t4, swz64(Yl, yr, 2 * tn + 1) + 2 * t4,
                  swz64(Yh, yr + 8, 2 * tn + 1) + 2 * t4, swz64(Yl, yr + 8, 2 * tn + 1) + 2 * t4, d1,
                  1.f);
    }
    __syncthreads();
    for (int t = warp; t < ntiles; t += PW) {
      const int p = t / per, tm = (t % per) / nb, tn = t % nb;
      const int s0 = 2 * bs * p;
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kb = 0; kb <= tm; ++kb) {  // X_D is lower triangular
        uint32_t ah[4], al[4], bh[4], bl[4];
        lda_rm_s(ah, sm.Fh, s0 + bs + 16 * tm, s0 + bs + 16 * kb, lane);
        lda_rm_s(al, sm.Fl, s0 + bs + 16 * tm, s0 + bs + 16 * kb, lane);
        ldb_kn_64(bh, Yh, p * bs + 16 * kb, 16 * tn, lane);
        ldb_kn_64(bl, Yl, p * bs + 16 * kb, 16 * tn, lane);
        mma_pair(d0, d1, ah, al, bh, bl);
      }
      const int fr = s0 + bs + 16 * tm + g4, fc = s0 + 16 * tn + 2 * t4;
      store_split(fel(sm.Fh, fr, fc), fel(sm.Fl, fr, fc), fel(sm.Fh, fr + 8, fc), fel(sm.Fl, fr + 8, fc),
                  d0, -1.f);
      store_split(fel(sm.Fh, fr, fc + 8), fel(sm.Fl, fr, fc + 8), fel(sm.Fh, fr + 8, fc + 8),
                  fel(sm.Fl, fr + 8, fc + 8), d1, -1.f);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(PT, 1) k_prep(PrepArgs a, const __grid_constant__ PrepMaps mp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  PrepSmem& sm = *reinterpret_cast<PrepSmem*>(base);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = a.Hv / a.Hk;
  const bool needP = a.P != nullptr, needU = a.U != nullptr, needW = a.W != nullptr;
  // TMEM row of this thread in the epilogues: lane quarter of the warp, column quarter
  const int quarter = warp & 3, cq = warp >> 2;
  const int row = 32 * quarter + lane;
  const long tile = (long)CH * CH;  // w, u and P tiles: [128][128] row-major in global memory
  // Persistent CTAs: this CTA's contiguous range of units (b, c, kh, jj), jj fastest
  const long U = (long)a.B * a.NC * a.Hk * group;
  const long u_begin = (long)blockIdx.x * U / gridDim.x, u_end = (long)(blockIdx.x + 1) * U / gridDim.x;
  struct Unit {
    int b, c, kh, jj;
  };
  auto decode = [&](long u) {  // 32-bit arithmetic: the unit count is below 2^31
    Unit x;
    const int uu = (int)u;
    x.jj = uu % group;
    const int gidx = uu / group;
    x.kh = gidx % a.Hk;
    const int ci = gidx / a.Hk;
    x.c = ci % a.NC;
    x.b = ci / a.NC;
    return x;
  };

  if (tid == 0) {
    tc::mbar_init(&sm.barKQ, 1);
    tc::mbar_init(&sm.barV[0], 1);
    tc::mbar_init(&sm.barV[1], 1);
    tc::mbar_init(&sm.barM, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::alloc(&sm.tmem, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  pdl_wait();     // the kernel before may still read the tiles this one overwrites
  pdl_release();
  const uint32_t tmem = sm.tmem;  // columns: K K^T 0, Q K^T 128, w 256, u 384
  const uint32_t tlane = tmem + ((uint32_t)(32 * quarter) << 16);
  bool ok = true;
  uint32_t mphase = 0;        // barM phases seen
  int kq_uses = 0;            // barKQ phases (one per key-head group)
  uint32_t v_use0 = 0, v_use1 = 0;  // barV[0], barV[1] phases

  // g and beta of row tid for unit u (loaded a head ahead; zero past the range or T)
  auto load_gates = [&](long u, float& gv, float& bv) {
    gv = bv = 0.f;
    if (u < u_end && tid < CH) {
      const Unit x = decode(u);
      if (tid < min(CH, a.T - x.c * CH)) {
        const long idx = ((long)x.b * a.T + x.c * CH + tid) * a.Hv + x.kh * group + x.jj;
        gv = act_g(a.g[idx], a.gate_logits);
        bv = act_beta(a.beta[idx], a.gate_logits);
      }
    }
  };
  float g_next = 0.f, b_next = 0.f;
  load_gates(u_begin, g_next, b_next);
  // The gate vectors of the value head that runs next (Gl = log2 of the chunk-local
  // cumsum, beta, etab); g_next, b_next hold its gates and are then reloaded with
  // those of unit u_after.  Warps 0-3 (a named barrier between them).
  auto build_gates = [&](long u_after) {
    if (tid < CH) {
      sm.Gl[tid] = g_next;
      sm.beta[tid] = b_next;
      load_gates(u_after, g_next, b_next);
      asm volatile("bar.sync 2, 128;" ::: "memory");
      if (warp == 0) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = sm.Gl[lane * 4 + i];
        warp_cumsum128(v, lane, a.c64 != 0);  // 64-token chunks: G restarts at row 64
#pragma unroll
        for (int i = 0; i < 4; ++i) sm.Gl[lane * 4 + i] = v[i] * LOG2E;
        __syncwarp();  // every Gl of the chunk is written (by this warp)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane * 4 + i;
          sm.etab[r] = exp2f(sm.Gl[r & ~15] - sm.Gl[r]);  // >= 1
        }
      }
    }
  };
  build_gates(u_begin + 1);  // the first value head's (read after the head's first barrier)
  unsigned char* const qbuf = reinterpret_cast<unsigned char*>(sm.Fh);
  // K and Q of the key-head group (b, c, kh): K into tile kbuf, Q into the Fh region
  auto load_kq = [&](int bb, int cc, int kk, unsigned char* kdst) {
    tc::arrive_expect_tx(&sm.barKQ, needP ? 2 * TILE : TILE);
    tc::tma_load_4d(kdst, &mp.k, 0, kk, cc * CH, bb, &sm.barKQ);
    tc::tma_load_4d(kdst + TILE / 2, &mp.k, 64, kk, cc * CH, bb, &sm.barKQ);
    if (needP) {
      tc::tma_load_4d(qbuf, &mp.q, 0, kk, cc * CH, bb, &sm.barKQ);
      tc::tma_load_4d(qbuf + TILE / 2, &mp.q, 64, kk, cc * CH, bb, &sm.barKQ);
    }
  };
  // V of value head j of (b, c) into tile dst, on barV[parity]
  auto load_v_to = [&](int bb, int cc, int j, unsigned char* dst, int parity) {
    uint64_t* bar = &sm.barV[parity];
    tc::arrive_expect_tx(bar, TILE);
    tc::tma_load_4d(dst, &mp.v, 0, j, cc * CH, bb, bar);
    tc::tma_load_4d(dst + TILE / 2, &mp.v, 64, j, cc * CH, bb, bar);
  };
  // Roles of the three tiles: K of the group in A[kb], V of the group's value
  // heads of even / odd position in A[vbi[0]] / A[vbi[1]].  During the last
  // value head of a group, the tile its predecessor's V used is free: the next
  // group's K goes there (and its Q into the Fh region once the inverse has
  // released it), so the next group starts with its K and Q already loaded;
  // its first two V go into the tiles the current group's K and last V held.
  int kb = 1, vbi[2] = {2, 0};
  bool next_loaded = false;     // K, Q (and the first V) of the next group already requested
  const int loader = 32;        // warp 1, lane 0: requests loads while thread 0 issues products

  for (long ug = u_begin; ug < u_end;) {
    // ---- a key-head group: value heads jj0 .. jj1 - 1 of (b, c, kh) -------------------
    const Unit x0 = decode(ug);
    const int c = x0.c, kh = x0.kh, b = x0.b, jj0 = x0.jj;
    const int jj1 = (int)min((long)group, jj0 + (u_end - ug));
    // V of value head kh * group + jj, the k-th head of the group, into its buffer
    auto load_v = [&](int jj) {
      const int k = jj - jj0;
      load_v_to(b, c, kh * group + jj, sm.A[vbi[k & 1]], k & 1);
    };
    // the next group of this CTA's range (valid if ug + jj1 - jj0 < u_end)
    const long ug_next = ug + (jj1 - jj0);
    const Unit xn = decode(ug_next < u_end ? ug_next : ug);
    if (tid == 0 && !next_loaded) {  // the first group of the range
      load_kq(b, c, kh, sm.A[kb]);
      if (needU) {
        load_v(jj0);
        if (jj0 + 1 < jj1) load_v(jj0 + 1);
      }
    }
    next_loaded = false;
    if (a.nrm) {
      // raw q and k: the rows' 1/||k|| and 1/||q||, 1 / sqrt(sum x^2 + 1e-6), go to
      // nrm (thread t: row t / 4, 32 columns).  The tiles stay raw, as the walk
      // reads them: K K^T, Q K^T and w = T'' K take the scales in their epilogues.
      ok = ok && tc::mbar_wait_sleep(&sm.barKQ, (uint32_t)(kq_uses & 1));
      float* nb = a.nrm + ((((long)b * a.Hk + kh) * a.NC + c) << 8);
      auto row_scale = [&](const unsigned char* tile, float* dst) {
        const int rr = tid >> 2, q4 = tid & 3;
        const unsigned char* rowp = tile + (q4 >> 1) * (TILE / 2) + rr * 128;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 x = *reinterpret_cast<const uint4*>(rowp + (((4 * (q4 & 1) + i) ^ (rr & 7)) << 4));
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16(w4[e]);
            ss += f.x * f.x + f.y * f.y;
          }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (q4 == 0) dst[rr] = rsqrtf(ss + 1e-6f);
      };
      row_scale(sm.A[kb], nb);
      if (needP) row_scale(qbuf, nb + CH);
      __syncthreads();  // the scales are read by every epilogue thread below
    }
    if (tid == 0) {
      ok = ok && tc::mbar_wait_sleep(&sm.barKQ, (uint32_t)(kq_uses & 1));
      tc::fence_after();
      tc::gemm_k128(tmem + 0, smem_u32(sm.A[kb]), smem_u32(sm.A[kb]), 128, false);
      if (needP) tc::gemm_k128(tmem + 128, smem_u32(qbuf), smem_u32(sm.A[kb]), 128, false);
      tc::commit(&sm.barM);
    }

    for (int jj = jj0; jj < jj1; ++jj) {
      const int j = kh * group + jj;
      const long bh = (long)b * a.Hv + j;
      const long chunk_id = bh * a.NC + c;
      const int vb = (jj - jj0) & 1;  // V buffer of this head
      // ---- gates of value head j: built while the previous head's products ran
      // the previous head's stores have read their staging tiles (Kg, Tp, F)
      // before the barrier below lets anyone rewrite them
      if (tid == 0 && (ug > u_begin || jj > jj0)) tc::bulk_wait_read();
      if (jj == jj0) {  // K K^T, Q K^T complete; K readable
        ok = ok && tc::mbar_wait_sleep(&sm.barKQ, (uint32_t)(kq_uses & 1));
        ok = ok && tc::mbar_wait_sleep(&sm.barM, mphase);
        mphase ^= 1;
        tc::fence_after();
      }
      if (tid == 0 && needU && jj > jj0 && jj + 1 < jj1)
        load_v(jj + 1);  // its buffer held V of head jj - 1, whose u is complete
      __syncthreads();

      // ---- S (hi/lo into F, fp32 diagonal blocks into Sd) and P (bf16 staging in Kg) ----
      // The decay exp2(Gl_r - Gl_s), s <= r, in a 16-column block starting at c0 is
      // exp2(Gl_r - Gl_c0) * etab[s]: G is non-increasing, so the first factor is
      // at most 1 and the second at least 1.  A block whose Gl drops by more than
      // 100 over its columns could overflow etab and takes the direct exponentials;
      // elsewhere a row whose first factor underflows has true decays below 2^-26.
      {
        const float Glr = sm.Gl[row];
        // raw K and Q rows: S takes 1/||k_r|| 1/||k_s||, P 1/||q_r|| 1/||k_s||
        const float* nb = a.nrm ? a.nrm + ((((long)b * a.Hk + kh) * a.NC + c) << 8) : nullptr;
        const float br = sm.beta[row] * (nb ? nb[row] : 1.f);
        const float pr = nb ? nb[CH + row] : 1.f;
        float* Sd = reinterpret_cast<float*>(sm.Tp + SD);
#pragma unroll 1
        for (int cb = 0; cb < 32; cb += 16) {
          const int c0 = 32 * cq + cb;
          float sv[16], pv[16];
          // warp-uniform: the block reaches the diagonal (and, with 64-token chunks,
          // lies in the rows' own chunk)
          if (c0 <= 32 * quarter + 31 && (!a.c64 || (c0 >> 6) == (quarter >> 1))) {
            float kk[16], mv[16];
            tc::ld16(tlane + c0, kk);
            if (needP) tc::ld16(tlane + 128 + c0, pv);
            if (sm.Gl[c0] - sm.Gl[c0 + 15] <= 100.f) {  // block-uniform
              const float fr = exp2f(Glr - sm.Gl[c0]);
#pragma unroll
              for (int i = 0; i < 16; ++i) mv[i] = fr * sm.etab[c0 + i];
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) mv[i] = exp2f(Glr - sm.Gl[c0 + i]);
            }
            if (nb) {
#pragma unroll
              for (int i = 0; i < 16; ++i) mv[i] *= nb[c0 + i];  // 1/||k_s|| of column s
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int s = c0 + i;
              const float m = (s <= row) ? mv[i] : 0.f;  // one decay for S and P
              sv[i] = (s < row) ? br * kk[i] * m : 0.f;
              pv[i] = needP ? pr * pv[i] * m : 0.f;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[i] = pv[i] = 0.f;
          }
          if (needP) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint4 o;
              o.x = pack_bf16(pv[8 * q + 0], pv[8 * q + 1]);
              o.y = pack_bf16(pv[8 * q + 2], pv[8 * q + 3]);
              o.z = pack_bf16(pv[8 * q + 4], pv[8 * q + 5]);
              o.w = pack_bf16(pv[8 * q + 6], pv[8 * q + 7]);
              *reinterpret_cast<uint4*>(sm.Kg + tc::sw128_chunk(row, (c0 >> 3) + q, CH)) = o;
            }
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint4 hi, lo;
            split8(sv + 8 * q, hi, lo);
            *reinterpret_cast<uint4*>(swz(sm.Fh, row, (c0 >> 3) + q)) = hi;
            *reinterpret_cast<uint4*>(swz(sm.Fl, row, (c0 >> 3) + q)) = lo;
          }
          if (((row >> 4) << 4) == c0) {  // this row's diagonal block, kept in fp32
            float* sd = Sd + (row >> 4) * 256 + (row & 15) * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<float4*>(sd + 4 * q) = make_float4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]);
          }
        }
      }
      tc::fence_proxy_async();  // P is read by a TMA store
      __syncthreads();
      if (tid == 0 && needP) {  // P leaves while the inverse runs
        const int y = (int)(chunk_id * CH);
        tc::tma_store_2d(&mp.P, 0, y, sm.Kg);
        tc::tma_store_2d(&mp.P, 64, y, sm.Kg + TILE / 2);
        tc::bulk_commit();
      }
      auto export_f32 = [&](float* dst) {
        for (int i = tid; i < CH * 16; i += PT) {
          const int r = i >> 4, jc = i & 15;
          float v[8];
          join8(*reinterpret_cast<const uint4*>(swz(sm.Fh, r, jc)), *reinterpret_cast<const uint4*>(swz(sm.Fl, r, jc)), v);
          *reinterpret_cast<float4*>(dst + r * CH + 8 * jc) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(dst + r * CH + 8 * jc + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
      };
      if (a.S_dbg) {
        export_f32(a.S_dbg + chunk_id * tile);
        __syncthreads();
      }

      // ---- T = (I + S)^-1 -------------------------------------------------------------
      if (a.c64)
        ut_inverse<64>(sm, warp, lane);
      else
        ut_inverse<CH>(sm, warp, lane);
      if (a.T_dbg) export_f32(a.T_dbg + chunk_id * tile);
      if (a.Tb) {
        bf16* dst = a.Tb + chunk_id * tile;
        for (int i = tid; i < CH * 16; i += PT) {
          const int r = i >> 4, jc = i & 15;
          float v[8];
          join8(*reinterpret_cast<const uint4*>(swz(sm.Fh, r, jc)), *reinterpret_cast<const uint4*>(swz(sm.Fl, r, jc)), v);
          uint4 o;
          o.x = pack_bf16(v[0], v[1]);
          o.y = pack_bf16(v[2], v[3]);
          o.z = pack_bf16(v[4], v[5]);
          o.w = pack_bf16(v[6], v[7]);
          *reinterpret_cast<uint4*>(dst + r * CH + 8 * jc) = o;
        }
      }
      // P's store has read Kg before T diag(beta gamma) is written there; the
      // decay table is dead, so it takes gamma (etab[s] = exp(G_s))
      // (with raw K rows also 1/||k_s||: T'' = T diag(beta gamma / ||k||), w = T'' K)
      if (tid < CH)
        sm.etab[tid] = exp2f(sm.Gl[tid]) * (a.nrm ? a.nrm[((((long)b * a.Hk + kh) * a.NC + c) << 8) + tid] : 1.f);
      if (tid == 0) tc::bulk_wait_read();
      __syncthreads();
      // ---- T' = T diag(beta) and T'' = T diag(beta gamma) (bf16, K-major SW128) ----------
      // u = T' V and w = T'' K: the gate of w folds into its A operand, so K
      // serves as w's B operand as loaded
#pragma unroll
      for (int i = 0; i < (CH * 16) / PT; ++i) {
        const int idx = tid + i * PT;
        const int r = idx >> 4, jc = idx & 15;
        float v[8];
        join8(*reinterpret_cast<const uint4*>(swz(sm.Fh, r, jc)), *reinterpret_cast<const uint4*>(swz(sm.Fl, r, jc)), v);
        const float4 b0 = *reinterpret_cast<const float4*>(&sm.beta[8 * jc]);
        const float4 b1 = *reinterpret_cast<const float4*>(&sm.beta[8 * jc + 4]);
        const float4 g0 = *reinterpret_cast<const float4*>(&sm.etab[8 * jc]);
        const float4 g1 = *reinterpret_cast<const float4*>(&sm.etab[8 * jc + 4]);
        const float tb[8] = {v[0] * b0.x, v[1] * b0.y, v[2] * b0.z, v[3] * b0.w,
                             v[4] * b1.x, v[5] * b1.y, v[6] * b1.z, v[7] * b1.w};
        const uint32_t off = tc::sw128_chunk(r, jc, CH);
        uint4 o;
        o.x = pack_bf16(tb[0], tb[1]);
        o.y = pack_bf16(tb[2], tb[3]);
        o.z = pack_bf16(tb[4], tb[5]);
        o.w = pack_bf16(tb[6], tb[7]);
        *reinterpret_cast<uint4*>(sm.Tp + off) = o;
        o.x = pack_bf16(tb[0] * g0.x, tb[1] * g0.y);
        o.y = pack_bf16(tb[2] * g0.z, tb[3] * g0.w);
        o.z = pack_bf16(tb[4] * g1.x, tb[5] * g1.y);
        o.w = pack_bf16(tb[6] * g1.z, tb[7] * g1.w);
        *reinterpret_cast<uint4*>(sm.Kg + off) = o;
      }
      tc::fence_proxy_async();
      tc::fence_before();
      __syncthreads();
      tc::fence_after();
      // ---- u = T' V,  w = T'' K -----------------------------------------------------------
      // the last value head of a group that has a successor in this CTA's range
      const bool last = (jj + 1 == jj1) && ug_next < u_end;
      if (tid == 0) {
        if (needU) {
          ok = ok && tc::mbar_wait_sleep(&sm.barV[vb], (vb ? v_use1 : v_use0) & 1u);
          tc::fence_after();
          tc::gemm_bmn_k128(tmem + 384, smem_u32(sm.Tp), smem_u32(sm.A[vbi[vb]]), false);
        }
        if (needW) tc::gemm_bmn_k128(tmem + 256, smem_u32(sm.Kg), smem_u32(sm.A[kb]), false);
        if (needU || needW) tc::commit(&sm.barM);
      }
      // the next group's K into the tile no V of this group needs any more, its Q
      // into the Fh region (the T' / T'' build has read it), while the products run
      if (tid == loader && last) load_kq(xn.b, xn.c, xn.kh, sm.A[vbi[(jj1 - jj0) & 1]]);
      // the next value head's gates, while the products run (this head's are dead)
      build_gates(ug + (jj - jj0) + 2);
      if (needU) (vb ? v_use1 : v_use0) += 1;
      if (needU || needW) {
        ok = ok && tc::mbar_wait_sleep(&sm.barM, mphase);
        mphase ^= 1;
        tc::fence_after();
      }
      if (last) {  // the products have read this group's K and last V: the next group's V go there
        if (tid == loader && needU) {
          const int jj1n = (int)min((long)group, xn.jj + (u_end - ug_next));
          load_v_to(xn.b, xn.c, xn.kh * group + xn.jj, sm.A[kb], 0);
          if (xn.jj + 1 < jj1n) load_v_to(xn.b, xn.c, xn.kh * group + xn.jj + 1, sm.A[vbi[vb]], 1);
        }
        const int kb_next = vbi[(jj1 - jj0) & 1];
        vbi[1] = vbi[vb];
        vbi[0] = kb;
        kb = kb_next;
        next_loaded = true;
      }
      // ---- w and u leave through shared staging tiles and TMA stores ------------------
      // (T'' and T' are dead now; their buffers hold w and u)
      if (needW) tmem_row_to_tile(tlane + 256 + 32 * cq, sm.Kg, row, cq);
      if (needU) tmem_row_to_tile(tlane + 384 + 32 * cq, sm.Tp, row, cq);
      tc::fence_proxy_async();
      tc::fence_before();
      __syncthreads();  // staging tiles complete; TMEM w/u and the gate vectors are free
      tc::fence_after();
      if (tid == 0 && (needW || needU)) {
        const int y = (int)(chunk_id * CH);
        if (needW) {
          tc::tma_store_2d(&mp.W, 0, y, sm.Kg);
          tc::tma_store_2d(&mp.W, 64, y, sm.Kg + TILE / 2);
        }
        if (needU) {
          tc::tma_store_2d(&mp.U, 0, y, sm.Tp);
          tc::tma_store_2d(&mp.U, 64, y, sm.Tp + TILE / 2);
        }
        tc::bulk_commit();
      }
    }
    ++kq_uses;
    ug += jj1 - jj0;
  }
  if (tid == 0) tc::bulk_wait();  // the stores have completed before the block exits
  if (!ok && a.status) atomicOr(a.status, 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

}  // namespace

size_t prep_smem_bytes() { return sizeof(PrepSmem) + 1024; }

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  PrepMaps mp;
  memset(&mp, 0, sizeof mp);
  if (!tmap_heads(&mp.k, a.k, a.B, a.T, a.Hk, HD)) return cudaErrorInvalidValue;
  if (a.P && !tmap_heads(&mp.q, a.q, a.B, a.T, a.Hk, HD)) return cudaErrorInvalidValue;
  if (a.U && !tmap_heads(&mp.v, a.v, a.B, a.T, a.Hv, HD)) return cudaErrorInvalidValue;
  const uint64_t rows = (uint64_t)a.B * a.Hv * a.NC * CH;
  if (a.W && !tmap_2d(&mp.W, a.W, HD, rows, HD * sizeof(bf16), 64, CH, true)) return cudaErrorInvalidValue;
  if (a.U && !tmap_2d(&mp.U, a.U, HD, rows, HD * sizeof(bf16), 64, CH, true)) return cudaErrorInvalidValue;
  if (a.P && !tmap_2d(&mp.P, a.P, CH, rows, CH * sizeof(bf16), 64, CH, true)) return cudaErrorInvalidValue;
  const size_t smem = prep_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // persistent CTAs, one per SM (the shared memory admits one), each taking a
  // contiguous range of (chunk, key head, value head) units
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long units = (long)a.B * a.NC * a.Hv;
  const int ctas = (int)(units < sms ? units : sms);
  if (ctas <= 0) return cudaSuccess;
  return launch_pdl(k_prep, dim3(ctas), dim3(PT), smem, s, a, mp);
}

}  // namespace gdn
