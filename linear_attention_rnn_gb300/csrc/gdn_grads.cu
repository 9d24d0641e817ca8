// gdn_grads.cu -- chunk-parallel gradients of the chunked gated delta rule.
//
// One CTA per (chunk c, key head, batch row b) serves the value heads j that
// share the key head, given for each the chunk's entering state h, the
// cotangent dh' of the state it leaves, Delta = u - w h and dDelta = P^T dO +
// k_g dh' (both stored by the two walks), and T.  Writing dV' = T^T dDelta,
// each line below reverses one line of the chunk forward:
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
//
// Every product is a 128 x 128 x 128 tcgen05 MMA into tensor memory (TMEM):
// dK and dQ of the key head accumulate there over its value heads (512
// columns: dK, dQ, and two scratch products), so dq and dk leave the CTA once,
// in bf16.  The row-scaled terms (-diag(beta gamma) dV' h^T, diag(ef) Delta
// dh'^T, diag(gamma) dO h^T) are formed by the epilogue threads from scratch
// products and written into the accumulators with tcgen05.st; the plain
// products (dKK K, dKK^T K, dQK^T Q, dQK K) then accumulate onto them.
// 16 warps: epilogue thread (row r, quarter cq) owns TMEM lane r, columns
// 32 cq .. 32 cq + 31.
// Operands are SW128 tiles: the stored tiles arrive by TMA, dV', dKK and dQK
// are written by the epilogues, and each product reads its tiles K-major or
// MN-major as the product needs (no transposes).
#include "gdn_kernels.cuh"
#include "gdn_tc05.cuh"
#include "gdn_tmap.cuh"

namespace gdn {

namespace {

constexpr uint32_t TILE = CH * HD * 2;
constexpr int GT = 512, GW = GT / 32;  // 16 warps
constexpr float LOG2E = 1.4426950408889634f;

struct GradSmem {
  unsigned char K[TILE], Q[TILE];  // SW128 [s][d] of the key head
  unsigned char W1[TILE];          // T; dV'; dKK
  unsigned char W2[TILE];          // dDelta; dh'; dO
  unsigned char W3[TILE];          // h
  unsigned char W4[TILE];          // Delta; dQK
  // per value head: its gates and per-row sums, two sets (by the parity of the
  // CTA's value-head count), so that a value head's gate cotangents can be
  // formed while the next value head starts
  struct HeadVec {
    float Gl[CH], gam[CH], ef[CH], beta[CH];
    float etab[CH];  // exp2(Gl[c0] - Gl[s]) for the 16-column block c0 of column s
    float colX[CH], dbeta[CH], dbg[CH], d_ef[CH], rowX[CH], dgamO[CH];
    float red[GW];
  } hv[2];
  float gcot[2][CH];  // a value head's dg and dbeta, formed by warp 15, stored later by it
  uint64_t barKQ, barT, barDD, barH, barDl, barDH, barDO, barM, barS8;
  uint32_t tmem;
};

// TMEM columns
constexpr uint32_t C_DK = 0, C_DQ = 128, C_A = 256, C_B = 384;

// Column sums over the 32 lanes of a warp: lane l holds 32 values of its own
// row; on return lane l holds the sum of column l (a reduce-scatter butterfly).
__device__ __forceinline__ float colsum32(float (&x)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? x[i] : x[i + w];
      const float keep = up ? x[i + w] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return x[0];
}

// 32 bf16 values (four 16-byte chunks) of row r, columns c0.., of a K-major SW128 tile
__device__ __forceinline__ void row32_load(const unsigned char* tile, int r, int c0, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + tc::sw128_chunk(r, (c0 >> 3) + q, CH));
    const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), c = unpack_bf16(u.z), d = unpack_bf16(u.w);
    v[8 * q + 0] = a.x;
    v[8 * q + 1] = a.y;
    v[8 * q + 2] = b.x;
    v[8 * q + 3] = b.y;
    v[8 * q + 4] = c.x;
    v[8 * q + 5] = c.y;
    v[8 * q + 6] = d.x;
    v[8 * q + 7] = d.y;
  }
}
__device__ __forceinline__ void row32_store(unsigned char* tile, int r, int c0, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 o;
    o.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
    o.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    o.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    o.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(tile + tc::sw128_chunk(r, (c0 >> 3) + q, CH)) = o;
  }
}
struct GradMaps {
  CUtensorMap k, q, dO, Tb, ddelta, states, delta, dstates;
  CUtensorMap dq, dk;  // stores over [B, T, Hk, 128] (rows past T are clipped)
};

__global__ void __launch_bounds__(GT, 1) k_grads(GradArgs a, const __grid_constant__ GradMaps mp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  GradSmem& sm = *reinterpret_cast<GradSmem*>(base);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = a.Hv / a.Hk;
  const int quarter = warp & 3, cq = warp >> 2;  // TMEM lane quarter, column quarter
  const int row = 32 * quarter + lane;
  // Persistent CTAs, one per SM, over contiguous ranges of (batch row, key head,
  // chunk) units, chunk fastest: a CTA pays its start-up once, and the tiles of
  // the next unit's first value head are requested while the current unit ends.
  const int U = a.B * a.Hk * a.NC;
  const int u_begin = (int)((long)blockIdx.x * U / gridDim.x);
  const int u_end = (int)((long)(blockIdx.x + 1) * U / gridDim.x);
  if (u_begin >= u_end) return;
  struct GUnit {
    int b, kh, c;
  };
  auto decode = [&](int u) {
    GUnit x;
    x.c = u % a.NC;
    const int r = u / a.NC;
    x.kh = r % a.Hk;
    x.b = r / a.Hk;
    return x;
  };
  auto cid_of = [&](const GUnit& x, int jj) { return ((long)x.b * a.Hv + x.kh * group + jj) * a.NC + x.c; };
  auto load2d = [&](unsigned char* dst, const CUtensorMap* m, long cid, uint64_t* bar) {
    tc::arrive_expect_tx(bar, TILE);
    tc::tma_load_2d(dst, m, 0, (int)(cid * CH), bar);
    tc::tma_load_2d(dst + TILE / 2, m, 64, (int)(cid * CH), bar);
  };
  auto load4d = [&](unsigned char* dst, const CUtensorMap* m, const GUnit& x, int head, uint64_t* bar) {
    tc::tma_load_4d(dst, m, 0, head, x.c * CH, x.b, bar);
    tc::tma_load_4d(dst + TILE / 2, m, 64, head, x.c * CH, x.b, bar);
  };
  auto load_kq = [&](const GUnit& x) {
    tc::arrive_expect_tx(&sm.barKQ, 2 * TILE);
    load4d(sm.K, &mp.k, x, x.kh, &sm.barKQ);
    load4d(sm.Q, &mp.q, x, x.kh, &sm.barKQ);
  };
  if (tid == 0) {
    tc::mbar_init(&sm.barKQ, 1);
    tc::mbar_init(&sm.barT, 1);
    tc::mbar_init(&sm.barDD, 1);
    tc::mbar_init(&sm.barH, 1);
    tc::mbar_init(&sm.barDl, 1);
    tc::mbar_init(&sm.barDH, 1);
    tc::mbar_init(&sm.barDO, 1);
    tc::mbar_init(&sm.barM, 1);
    tc::mbar_init(&sm.barS8, 1);
    tc::mbar_fence_init();
    // the first unit's K, Q (inputs) and T (written by the preparation, which
    // completed before the kernel just before this one started)
    const GUnit x0 = decode(u_begin);
    load_kq(x0);
    load2d(sm.W1, &mp.Tb, cid_of(x0, 0), &sm.barT);
  }
  // dDelta, dh' and (without a saved buffer) the entering states and Delta come
  // from the kernel just before; every store follows too
  pdl_wait();
  pdl_release();
  if (tid == 0) {
    const long cid0 = cid_of(decode(u_begin), 0);
    load2d(sm.W2, &mp.ddelta, cid0, &sm.barDD);
    load2d(sm.W3, &mp.states, cid0, &sm.barH);
    load2d(sm.W4, &mp.delta, cid0, &sm.barDl);
  }
  if (warp == 0) tc::alloc(&sm.tmem, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16) + 32u * cq;  // lane row, column quarter
  const int c0 = 32 * cq;
  bool ok = true;
  uint32_t mc = 0;  // completed-commit count of barM seen by this thread
  auto wait_mma = [&]() {
    ok = ok && tc::mbar_wait_sleep(&sm.barM, mc & 1);
    ++mc;
    tc::fence_after();
  };
  auto sync_operands = [&]() {  // epilogue-written operand tiles -> tensor core
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  };
  // raw g and beta of row tid for value head jj of unit x (loaded a head ahead,
  // straight into their registers: activated where they are used, a head later)
  auto load_gates = [&](const GUnit& x, int jj, float& gv, float& bv) {
    gv = bv = 0.f;
    const bool in = tid < min(CH, a.T - x.c * CH);
    const long idx = ((long)x.b * a.T + x.c * CH + (in ? tid : 0)) * a.Hv + x.kh * group + jj;
    ld_pred_f32(gv, a.g + idx, in);
    ld_pred_f32(bv, a.beta + idx, in);
  };
  float g_next = 0.f, b_next = 0.f;
  if (tid < CH) load_gates(decode(u_begin), 0, g_next, b_next);
  // Gate cotangents of a value head (one warp): dg = reverse cumsum over the chunk
  // of dG, dbeta; with gate logits the chain rule through the activations.  They
  // are formed into sm.gcot (gate_cot) and written out by gate_cot_store, later:
  // at a value head's start the memory pipe is full of that head's V-row loads,
  // and stores issued then wait behind them.
  auto gate_cot = [&](const GradSmem::HeadVec& P, int L_p) {
    float dgC = 0.f;
#pragma unroll
    for (int w = 0; w < GW; ++w) dgC += P.red[w];
    float sum_def = 0.f;
    float dG[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      const float de = P.d_ef[r] * P.ef[r];
      sum_def += de;
      const float dgam = P.dgamO[r] + P.beta[r] * P.dbg[r];
      dG[i] = P.gam[r] * dgam + P.rowX[r] - P.colX[r] - de;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum_def += __shfl_xor_sync(0xffffffffu, sum_def, off);
    if (lane == 31) dG[3] += P.gam[CH - 1] * dgC + sum_def;  // row C-1: gamma_C = gamma[C-1]
    // reverse inclusive cumsum over the 128 rows: dg_s = sum_{r >= s} dG_r
    const float tot = dG[0] + dG[1] + dG[2] + dG[3];
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
      sm.gcot[0][r] = dg[i];
      sm.gcot[1][r] = P.dbeta[r] + P.gam[r] * P.dbg[r];
    }
    // (no warp barrier: the warp reads sm.gcot back only after several CTA barriers,
    // and one here would wait for its outstanding V-row loads)
    (void)L_p;
  };
  auto gate_cot_store = [&](long tokv_p, int L_p) {  // the same warp, after gate_cot
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane + 32 * i;
      if (r < L_p) {
        const long t = tokv_p + (long)r * a.Hv;
        float dgv = sm.gcot[0][r], dbv = sm.gcot[1][r];
        if (a.gate_logits) {  // chain rule through g = -softplus(a) and beta = sigmoid(b)
          const float sa = act_beta(a.g[t], 1), sb = act_beta(a.beta[t], 1);
          dgv *= -sa;
          dbv *= sb * (1.f - sb);
        }
        a.dg[t] = dgv;
        a.dbeta[t] = dbv;
      }
    }
  };
  bool kq_pending = false;  // thread 0: the unit's K and Q are still to be requested
  long pend_tokv = 0;  // the value head whose gate cotangents are pending
  int pend_L = 0;
  int hc = 0;  // value heads processed by this CTA: the parity of the tile barriers

  for (int u = u_begin; u < u_end; ++u) {
  const GUnit xu = decode(u);
  const int c = xu.c, kh = xu.kh, b = xu.b;
  const int t0 = c * CH;
  const int L = min(CH, a.T - t0);
  const bool has_next = u + 1 < u_end;
  const GUnit xn = decode(has_next ? u + 1 : u);
  const uint32_t kq_par = (uint32_t)((u - u_begin) & 1);
  for (int jj = 0; jj < group; ++jj) {
    const int j = kh * group + jj;
    const long cid = cid_of(xu, jj);
    const long tokv = ((long)b * a.T + t0) * a.Hv + j;  // row 0 of the v/dO tile
    const uint32_t par = (uint32_t)(hc & 1);
    GradSmem::HeadVec& H = sm.hv[hc & 1];
    // the value head after this one: the next of this unit, or the next unit's first
    const bool next_here = jj + 1 < group;
    const bool has_after = next_here || has_next;
    const long cid_after = next_here ? cid_of(xu, jj + 1) : cid_of(xn, 0);
    // this head's V rows for the dv pass (warps 4-15, 16 threads per 256-byte row),
    // requested now so that their latency passes under S1 and E1.  Warps 0-3 build
    // the gates behind two barriers, and a barrier waits for the loads its threads
    // have outstanding: they load none.
    constexpr int DW0 = 4;                       // first warp of the dv pass
    constexpr int DT = GT - 32 * DW0;            // 384 threads
    constexpr int NI = (CH * 16 + DT - 1) / DT;  // 6 passes (the last one for warps 4-7 only)
    uint4 v4[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int idx = tid - 32 * DW0 + i * DT;
      const int r = idx >> 4, jc = idx & 15;
      const bool in = warp >= DW0 && idx < CH * 16 && r < L;
      v4[i] = make_uint4(0u, 0u, 0u, 0u);
      ld_pred_v4(v4[i], a.v + (tokv + (long)(in ? r : 0) * a.Hv) * HD + 8 * (in ? jc : 0), in);
    }
    // ---- gates of value head j; per-row sums cleared ----------------------------
    // (meanwhile warp 15 forms the previous value head's gate cotangents, and warp
    // 14 issues S1 once T and dDelta are in and then requests Delta once the
    // previous head's S8b has read W4; the two barriers of this part are over warps
    // 0-3, which write and scan the gates; the other warps read them after E1's barrier)
    if (warp == GW - 1) {
      if (hc > 0) gate_cot(sm.hv[(hc - 1) & 1], pend_L);
    } else if (tid == 32 * (GW - 2)) {  // S1: dV' = T^T dDelta (both tiles read MN-major)
      ok = ok && tc::mbar_wait(&sm.barT, par);
      ok = ok && tc::mbar_wait(&sm.barDD, par);
      tc::fence_after();
      tc::gemm128(tmem + C_A, smem_u32(sm.W1), true, smem_u32(sm.W2), true, false);
      tc::commit(&sm.barM);
      if (hc > 0) {  // (the first value head's Delta came with the CTA's first tiles)
        ok = ok && tc::mbar_wait(&sm.barS8, (uint32_t)((hc - 1) & 1));
        load2d(sm.W4, &mp.delta, cid, &sm.barDl);
      }
    }
    if (tid < CH) {
      H.Gl[tid] = tid < L ? act_g(g_next, a.gate_logits) : 0.f;
      H.beta[tid] = tid < L ? act_beta(b_next, a.gate_logits) : 0.f;
      if (next_here)
        load_gates(xu, jj + 1, g_next, b_next);
      else if (has_next)
        load_gates(xn, 0, g_next, b_next);
      H.colX[tid] = H.dbeta[tid] = H.dbg[tid] = H.d_ef[tid] = H.rowX[tid] = H.dgamO[tid] = 0.f;
    }
    if (warp < 4) asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == 0) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = H.Gl[lane * 4 + i];
      warp_cumsum128(v, lane);
      const float Glast = __shfl_sync(0xffffffffu, v[3], 31);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane * 4 + i;
        H.Gl[r] = v[i] * LOG2E;
        H.gam[r] = expf(v[i]);
        H.ef[r] = expf(Glast - v[i]);
      }
      __syncwarp();  // every Gl of the chunk is written (by this warp)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = lane * 4 + i;
        H.etab[r] = exp2f(H.Gl[r & ~15] - H.Gl[r]);  // >= 1
      }
    }
    if (warp < 4) asm volatile("bar.sync 1, 128;" ::: "memory");
    if (tid == 0 && kq_pending) {  // the last unit's dq, dk stores have read the K, Q tiles
      tc::bulk_wait_read();
      load_kq(xu);
      kq_pending = false;
    }
    // this row's gates, read after E1's barrier (which warps 14 and 15 reach late)
    float Glr = 0.f, br = 0.f, gr = 0.f, efr = 0.f, bgr = 0.f;
    float p_db = 0.f, p_dbg = 0.f, p_def = 0.f, p_rowx = 0.f, p_dgam = 0.f;
    // Decays exp2(Gl_r - Gl_s) of columns c0..c0+31 of this thread's row, masked to
    // s < r (or s <= r).  G is non-increasing, so in each 16-column block b0 the decay
    // is exp2(Gl_r - Gl_b0) (at most 1) times etab[s] (at least 1); a block whose Gl
    // drops by more than 100 could overflow etab and takes the direct exponentials.
    auto fill_decay = [&](int c0, float (&m)[32], bool incl) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b0 = c0 + 16 * h;
        if (H.Gl[b0] - H.Gl[b0 + 15] <= 100.f) {  // block-uniform
          const float fr = exp2f(Glr - H.Gl[b0]);
#pragma unroll
          for (int i = 0; i < 16; ++i) m[16 * h + i] = fr * H.etab[b0 + i];
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) m[16 * h + i] = exp2f(Glr - H.Gl[b0 + i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int s = c0 + i;
        m[i] = (incl ? s <= row : s < row) ? m[i] : 0.f;
      }
    };

    // ---- E1: dV' -> W1 (bf16) ------------------------------------------------------------
    wait_mma();
    if (tid == 0) load2d(sm.W2, &mp.dstates, cid, &sm.barDH);  // dDelta has been read
    {
      float x[32];
      tc::ld32(tl + C_A, x);
      row32_store(sm.W1, row, c0, x);
    }
    sync_operands();
    Glr = H.Gl[row];
    br = H.beta[row];
    gr = H.gam[row];
    efr = H.ef[row];
    bgr = br * gr;

    // ---- S2: dV' h^T -> A;  S5: Delta dh'^T -> B --------------------------------------
    if (tid == 0) {
      ok = ok && tc::mbar_wait(&sm.barH, par);
      ok = ok && tc::mbar_wait(&sm.barDl, par);
      ok = ok && tc::mbar_wait(&sm.barDH, par);
      tc::fence_after();
      tc::gemm128(tmem + C_A, smem_u32(sm.W1), false, smem_u32(sm.W3), false, false);
      tc::gemm128(tmem + C_B, smem_u32(sm.W4), false, smem_u32(sm.W2), false, false);
      tc::commit(&sm.barM);
    }
    // ---- dv = diag(beta) dV' and dbeta += rowsum(dV' V), while S2/S5 run -----------------
    // Read back from the bf16 dV' tile with 16 threads per row, so that V is
    // loaded and dv stored in whole 256-byte rows.  Warps 0-3 take no share: warp
    // 0's thread 0 waits for dh' and issues S2/S5 meanwhile (a share of its own
    // would put that wait in front of every later barrier), and warps 0-3 hold no
    // V loads at the gates' barriers.  384 threads, 24 rows' worth of 16-byte
    // chunks per pass (a 16-lane group stays on one row).
    if (warp >= DW0) {
      const int t2 = tid - 32 * DW0;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int idx = t2 + i * DT;
        if (idx >= CH * 16) break;  // warp-uniform: whole warps run out together
        const int r = idx >> 4, jc = idx & 15;
        const uint4 d4 = *reinterpret_cast<const uint4*>(sm.W1 + tc::sw128_chunk(r, jc, CH));
        const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w}, vw[4] = {v4[i].x, v4[i].y, v4[i].z, v4[i].w};
        const float bt = H.beta[r];
        float part = 0.f;
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 dd = unpack_bf16(dw[e]), vv = unpack_bf16(vw[e]);
          part += dd.x * vv.x + dd.y * vv.y;
          ow[e] = pack_bf16(bt * dd.x, bt * dd.y);
        }
        if (r < L)
          *reinterpret_cast<uint4*>(a.dv + (tokv + (long)r * a.Hv) * HD + 8 * jc) =
              make_uint4(ow[0], ow[1], ow[2], ow[3]);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if ((lane & 15) == 0) atomicAdd(&H.dbeta[r], part);
      }
    }
    {  // <dh', h>: elementwise over two tiles of the same layout
      ok = ok && tc::mbar_wait_sleep(&sm.barDH, par);
      ok = ok && tc::mbar_wait_sleep(&sm.barH, par);
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < (int)(TILE / 16) / GT; ++i) {
        const uint32_t off = (uint32_t)(tid + i * GT) * 16u;
        const uint4 x = *reinterpret_cast<const uint4*>(sm.W2 + off);
        const uint4 y = *reinterpret_cast<const uint4*>(sm.W3 + off);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 p = unpack_bf16(xs[e]), q = unpack_bf16(ys[e]);
          d += p.x * q.x + p.y * q.y;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (lane == 0) H.red[warp] = d;
    }

    // ---- E2: dK (+)= -diag(beta gamma) dV' h^T + diag(ef) Delta dh'^T ---------------------
    if (jj == 0) ok = ok && tc::mbar_wait_sleep(&sm.barKQ, kq_par);  // the unit's K and Q (read from here on)
    wait_mma();
    {
      float kv[32], x[32], acc[32];
      row32_load(sm.K, row, c0, kv);
      if (jj > 0) {
        tc::ld32(tl + C_DK, acc);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      }
      tc::ld32(tl + C_A, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p_dbg -= x[i] * kv[i];
        acc[i] -= bgr * x[i];
      }
      tc::ld32(tl + C_B, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p_def += x[i] * kv[i];
        acc[i] += efr * x[i];
      }
      tc::st32(tl + C_DK, acc);
    }
    tc::wait_st();
    tc::fence_before();
    __syncthreads();  // also: every thread is done with dh' (W2)
    tc::fence_after();

    // ---- S3: ds = dV' Delta^T -> A;  K K^T -> B ----------------------------------------
    if (tid == 0) {
      tc::arrive_expect_tx(&sm.barDO, TILE);
      load4d(sm.W2, &mp.dO, xu, j, &sm.barDO);
      tc::gemm128(tmem + C_A, smem_u32(sm.W1), false, smem_u32(sm.W4), false, false);
      tc::gemm128(tmem + C_B, smem_u32(sm.K), false, smem_u32(sm.K), false, false);
      tc::commit(&sm.barM);
    }
    // ---- E3: dKK = -(ds * M) diag-row(beta), strictly lower -> W1; dbeta, rowX, colX -----
    // (warp 15: the previous value head's gate cotangents leave while S3 runs)
    if (warp == GW - 1 && hc > 0) gate_cot_store(pend_tokv, pend_L);
    wait_mma();
    {
      float out[32];
      if (cq <= quarter) {  // warp-uniform: the block reaches the diagonal
        float ds[32], kk[32];
        tc::ld32(tl + C_A, ds);
        tc::ld32(tl + C_B, kk);
        fill_decay(c0, out, false);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float M = out[i];  // 0 off the strict lower triangle
          const float dS = -ds[i];
          p_db += dS * kk[i] * M;
          const float dkk = dS * br * M;
          out[i] = dkk;
          ds[i] = dkk * kk[i];
          p_rowx += ds[i];
        }
        const float cs = colsum32(ds, lane);
        atomicAdd(&H.colX[c0 + lane], cs);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) out[i] = 0.f;
      }
      row32_store(sm.W1, row, c0, out);
    }
    sync_operands();

    // ---- S4: dK += dKK K + dKK^T K;  S6: dP = dO Delta^T -> A;  Q K^T -> B -------------
    // (S6 first and committed alone: E4 needs only it, and S4 runs under E4)
    if (tid == 0) {
      ok = ok && tc::mbar_wait(&sm.barDO, par);
      tc::fence_after();
      tc::gemm128(tmem + C_A, smem_u32(sm.W2), false, smem_u32(sm.W4), false, false);
      tc::gemm128(tmem + C_B, smem_u32(sm.Q), false, smem_u32(sm.K), false, false);
      tc::commit(&sm.barM);
      tc::gemm128(tmem + C_DK, smem_u32(sm.W1), false, smem_u32(sm.K), true, true);
      tc::gemm128(tmem + C_DK, smem_u32(sm.W1), true, smem_u32(sm.K), true, true);
    }
    // ---- E4: dQK = dP * M (diagonal included) -> W4; rowX, colX --------------------------
    wait_mma();
    {
      float out[32];
      if (cq <= quarter) {
        float dp[32], qk[32];
        tc::ld32(tl + C_A, dp);
        tc::ld32(tl + C_B, qk);
        fill_decay(c0, out, true);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float M = out[i];  // 0 above the diagonal
          const float d = dp[i] * M;
          out[i] = d;
          dp[i] = d * qk[i];
          p_rowx += dp[i];
        }
        const float cs = colsum32(dp, lane);
        atomicAdd(&H.colX[c0 + lane], cs);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) out[i] = 0.f;
      }
      row32_store(sm.W4, row, c0, out);
    }
    sync_operands();

    // ---- S7: dK += dQK^T Q;  S8: dO h^T -> A -------------------------------------------
    // (S8 first and committed alone: E5 needs only it, and S7 runs under E5; the
    // commit also covers S4, issued before it, so W1 may be reloaded at E5)
    if (tid == 0) {
      tc::gemm128(tmem + C_A, smem_u32(sm.W2), false, smem_u32(sm.W3), false, false);
      tc::commit(&sm.barM);
      tc::gemm128(tmem + C_DK, smem_u32(sm.W4), true, smem_u32(sm.Q), true, true);
    }
    // ---- E5: dgamma_O = rowsum(Q * (dO h^T));  dQ (+)= diag(gamma) dO h^T ------------------
    wait_mma();
    if (tid == 0 && has_after) {  // next value head: its T, dDelta, h (tiles consumed)
      load2d(sm.W1, &mp.Tb, cid_after, &sm.barT);
      load2d(sm.W2, &mp.ddelta, cid_after, &sm.barDD);
      load2d(sm.W3, &mp.states, cid_after, &sm.barH);
    }
    {
      float qv[32], x[32], acc[32];
      row32_load(sm.Q, row, c0, qv);
      tc::ld32(tl + C_A, x);
      if (jj > 0) {
        tc::ld32(tl + C_DQ, acc);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p_dgam += x[i] * qv[i];
        acc[i] += gr * x[i];
      }
      tc::st32(tl + C_DQ, acc);
    }
    tc::wait_st();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // ---- S8b: dQ += dQK K ----------------------------------------------------------------
    // (committed to barS8, covering S7 too: waited for before W4 is reloaded, by
    // warp 14 at the next value head's start, and before the unit's dq, dk leave)
    if (tid == 0) {
      tc::gemm128(tmem + C_DQ, smem_u32(sm.W4), false, smem_u32(sm.K), true, true);
      tc::commit(&sm.barS8);
    }
    atomicAdd(&H.dbeta[row], p_db);
    atomicAdd(&H.dbg[row], p_dbg);
    atomicAdd(&H.d_ef[row], p_def);
    atomicAdd(&H.rowX[row], p_rowx);
    atomicAdd(&H.dgamO[row], p_dgam);
    // (its gate cotangents: warp 15, at the next value head's start)
    pend_tokv = tokv;
    pend_L = L;
    __syncthreads();
    ++hc;
  }

  // ---- dq, dk of the key head: bf16 staging tiles in the Q and K buffers, once the
  //      unit's last products (S7, S8b) have completed and read them; W1-W3 already
  //      hold the next unit's first tiles ------------------------------------------------
  ok = ok && tc::mbar_wait_sleep(&sm.barS8, (uint32_t)((hc - 1) & 1));
  tc::fence_after();
  {
    float x[32];
    tc::ld32(tl + C_DQ, x);
    row32_store(sm.Q, row, c0, x);
    tc::ld32(tl + C_DK, x);
    row32_store(sm.K, row, c0, x);
  }
  tc::fence_proxy_async();
  __syncthreads();
  if (tid == 0) {
    tc::tma_store_4d(&mp.dq, 0, kh, t0, b, sm.Q);
    tc::tma_store_4d(&mp.dq, 64, kh, t0, b, sm.Q + TILE / 2);
    tc::tma_store_4d(&mp.dk, 0, kh, t0, b, sm.K);
    tc::tma_store_4d(&mp.dk, 64, kh, t0, b, sm.K + TILE / 2);
    tc::bulk_commit();
    // (the next unit's K and Q are requested once these stores have read the staging
    // tiles: at the next value head's start, after its gates, where thread 0 waits
    // for S1 anyway; waiting here held warp 0, and with it the next head's start)
    kq_pending = has_next;
  }
  }  // units
  if (warp == GW - 1 && hc > 0) {
    gate_cot(sm.hv[(hc - 1) & 1], pend_L);
    gate_cot_store(pend_tokv, pend_L);
  }
  if (tid == 0) tc::bulk_wait();  // every store has completed before the block exits
  if (!ok && a.status) atomicOr(a.status, 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

}  // namespace

size_t grad_smem_bytes() { return sizeof(GradSmem) + 1024; }

cudaError_t launch_grads(const GradArgs& a, cudaStream_t s) {
  GradMaps mp;
  memset(&mp, 0, sizeof mp);
  const uint64_t rows = (uint64_t)a.B * a.Hv * a.NC * CH;
  bool ok = tmap_heads(&mp.k, a.k, a.B, a.T, a.Hk, HD) && tmap_heads(&mp.q, a.q, a.B, a.T, a.Hk, HD) &&
            tmap_heads(&mp.dO, a.dO, a.B, a.T, a.Hv, HD);
  ok = ok && tmap_2d(&mp.Tb, a.Tb, CH, rows, CH * 2, 64, CH, true);
  ok = ok && tmap_2d(&mp.ddelta, a.ddelta, HD, rows, HD * 2, 64, CH, true);
  ok = ok && tmap_2d(&mp.states, a.states, HD, rows, HD * 2, 64, CH, true);
  ok = ok && tmap_2d(&mp.delta, a.delta, HD, rows, HD * 2, 64, CH, true);
  ok = ok && tmap_2d(&mp.dstates, a.dstates, HD, rows, HD * 2, 64, CH, true);
  ok = ok && tmap_heads(&mp.dq, a.dq, a.B, a.T, a.Hk, HD) && tmap_heads(&mp.dk, a.dk, a.B, a.T, a.Hk, HD);
  if (!ok) return cudaErrorInvalidValue;
  const size_t smem = grad_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(k_grads, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // persistent CTAs, one per SM (the shared memory admits one), each over a
  // contiguous range of (batch row, key head, chunk) units
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long units = (long)a.B * a.Hk * a.NC;
  const int ctas = (int)(units < sms ? units : sms);
  if (ctas <= 0) return cudaSuccess;
  return launch_pdl(k_grads, dim3(ctas), dim3(GT), smem, s, a, mp);
}

}  // namespace gdn
