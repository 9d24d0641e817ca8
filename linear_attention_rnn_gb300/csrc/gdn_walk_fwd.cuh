// gdn_walk_fwd.cuh -- sequential forward walk over the chunks of a segment
// (device body; the kernels that run it are in gdn_walk_fwd.cu and gdn_walk_pair.cu).
//
// Inter-chunk step ("GatedDeltaNet does not support ici_context_parallelism",
// section "The recurrence is affine, so it can be parallelized"):
//     Delta = u - w h,     h' = exp(g_last) h + k_g^T Delta,
// with k_g = diag(exp(G_last - G)) K, and the masked intra-chunk output
//     O = diag(gamma) Q h + P Delta,      P = (Q K^T) * decay (diagonal included).
//
// One CTA walks a slice of SW = 32 or 64 columns of one head's state (columns
// of h evolve independently: every matrix of the step acts on h from the
// left).  Compute thread (r, g) owns row r, columns 32 g .. 32 g + 31 of the
// slice in fp32 registers for the whole segment, and those columns of TMEM
// lane r in every product.  Per chunk the products
//     X  = w h            (A = w, K-major)
//     H' = K^T (ef Delta) (A = the K tile read MN-major: no transpose pass)
//     O1 = Q h,  O2 = P Delta
// are tcgen05 MMAs (M = 128, N = SW, K = 128) into tensor memory.  Their B
// operands (h^T, Delta^T, (ef Delta)^T, SW x 128 bf16) are written column by
// column by the compute threads in the 128-byte-swizzled K-major layout.
//
// Warp roles after the compute warps: a chain issuer (X, H' as soon as their
// operands are signalled ready on mbarriers), a TMA producer (the chunk tiles
// w, Q, K, P in the order consumed, into a ring of 32 KiB slots, each refilled
// as soon as the MMA that read it has completed), and a third warp that, in
// the output mode, issues O1 and O2 (so that their issue never holds the
// chain's issuer) and, in the recompute mode, stores the staged exports.  A
// TMA request can block its thread while earlier copies stream in, so the
// loads never share a thread with an MMA issuer.  Each compute thread reads
// its row of the u slice straight into registers a chunk ahead.  The compute
// threads never wait on memory issue, only on MMA completion.  Every wait is
// bounded; one that gives up sets bit 0 of the status word.
//
// Modes:
//   RECUR (fold = 0): walk from the segment's entering state, write O (if o
//     is given), and optionally (STAGED) the bf16 entering state and Delta of
//     every chunk, for the backward, and the final state (last segment).  With
//     both output and exports the tile ring has one slot fewer (the last one
//     stages the exports) and a fourth extra warp stores them.
//   FOLD  (fold = 1): pass 1 of the two-pass segment scan ("Shard the
//     GatedDeltaNet sequence under ici_context_parallelism", description):
//     push the augmented state [A | B] through the segment's chunks starting
//     from [I | 0]; the A columns take no u term.  CTAs 0-3 hold A's column
//     slices, 4-7 hold B's.
//
// 64-token chunks (C64; RECUR without exports, and FOLD): the state steps every
// 64 tokens and each step keeps 128-row products.  The first product's A
// operand stacks the chunk's w (rows 0-63) over its Q (rows 64-127), so one
// product gives both w h (TMEM lanes 0-63) and Q h (lanes 64-127).  Compute
// threads of rows 0-63 form Delta, whose images hold 64 K-columns; the state
// update K^T (ef Delta) and P Delta take K = 64, and P Delta's A operand holds
// the chunk's 64 x 64 P in rows 64-127, so that the output rows meet Q h in
// lanes 64-127, where the threads of rows 64-127 write them.
#pragma once
#include "gdn_kernels.cuh"
#include "gdn_tc05.cuh"

namespace gdn {
namespace walkf {

constexpr uint32_t TILE_BYTES = CH * HD * 2;  // 32 KiB

// Layout per slice width SW (state columns per CTA: 32 or 64)
template <int SW>
struct FwdCfg {
  static constexpr int NCT = 4 * SW;               // compute threads: 4 lane quarters x SW / 32 column groups
  static constexpr int NCW = NCT / 32;             // compute warps
  static constexpr int NT = NCT + 96;              // + MMA issuer, TMA producer and TMA store warps
  static constexpr int NSLOT = SW == 32 ? 6 : 5;   // tile ring slots (the last one doubles as staging)
  static constexpr int NSTAGE = SW == 32 ? 2 : 1;  // staging sets of the exported h and Delta slices
  static constexpr uint32_t BT = SW * HD * 2;      // a [SW x 128] B-operand image
  static constexpr uint32_t SLICE = CH * SW * 2;   // a [128 x SW] staged slice
  static constexpr uint32_t TMEM_COLS = SW == 32 ? 256 : 512;  // X, H', two O1, O2: 5 SW columns
};

template <int SW>
struct WalkSmem {
  using C = FwdCfg<SW>;
  unsigned char slot[C::NSLOT][TILE_BYTES];
  unsigned char Ht[2][C::BT];  // h^T of chunk index i in Ht[i & 1]
  unsigned char Dt[C::BT];
  unsigned char Dgt[C::BT];
  float gsum[2][4];
  uint64_t full[C::NSLOT], empty[C::NSLOT];
  uint64_t barX, barO1, barH, barO2, barDg, barD, barHt;
  uint64_t sfull[2], sempty[2];  // staging set: written by the compute threads / read by its stores
  uint32_t tmem;
};

// Column k of a [SW x 128] K-major SW128 B image: rows n0 .. n0 + 31 from 32 fp32 values.
template <int SW>
__device__ __forceinline__ void write_bt_column(unsigned char* tile, int k, int n0, const float (&v)[32]) {
#pragma unroll
  for (int n = 0; n < 32; ++n)
    *reinterpret_cast<bf16*>(tile + tc::sw128(n0 + n, k, SW)) = __float2bfloat16_rn(v[n]);
}

__device__ __forceinline__ void store_row_bf16(bf16* dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 o;
    o.x = pack_bf16(v[8 * q], v[8 * q + 1]);
    o.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    o.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    o.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(dst + 8 * q) = o;
  }
}

// row r, columns 32 g .. 32 g + 31 of a [128 x SW] staged slice (SW 32: 64-byte
// swizzle; SW 64: 128-byte swizzle, the layouts the slices' tensor maps store)
template <int SW>
__device__ __forceinline__ void stage_row(unsigned char* buf, int r, int g, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 o;
    o.x = pack_bf16(v[8 * q], v[8 * q + 1]);
    o.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    o.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    o.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    const uint32_t off = SW == 32 ? tc::sw64_chunk(r, q) : (uint32_t)(r * 128 + (((4 * g + q) ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(buf + off) = o;
  }
}

__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The walk of CTA (slice, seg, bhi) with FwdCfg<SW>::NT threads; `base` is the
// 1024-byte-aligned dynamic shared memory (sizeof(WalkSmem<SW>) bytes).
// STAGED: the recompute mode (exports h and Delta, no output).
template <bool FOLD, bool STAGED, int SW, bool C64 = false>
__device__ __forceinline__ void walk(const WalkFwdArgs& a, const WalkFwdMaps& mp, unsigned char* base, int slice,
                                     int seg, int bhi) {
  static_assert(!(C64 && STAGED), "64-token chunks export nothing");
  constexpr int CC = C64 ? 64 : CH;  // tokens per chunk
  using Cfg = FwdCfg<SW>;
  constexpr int NCT = Cfg::NCT, NCW = Cfg::NCW, NSLOT = Cfg::NSLOT, NSTAGE = Cfg::NSTAGE;
  constexpr uint32_t SLICE = Cfg::SLICE;
  constexpr int NSL = HD / SW;  // slices per state
  WalkSmem<SW>& sm = *reinterpret_cast<WalkSmem<SW>*>(base);
  const int b = bhi / a.Hv, j = bhi % a.Hv, kh = j / (a.Hv / a.Hk);
  const long bh = bhi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cbeg = (int)((long)seg * a.NC / a.S), cend = (int)((long)(seg + 1) * a.NC / a.S);
  const bool partA = FOLD && slice < NSL;  // A columns: no u term
  const bool withO = !FOLD && a.o != nullptr;
  // tiles per chunk: w, (Q,) K (, P); with 64-token chunks [w; Q] (or w), K (, P)
  const int TPC = withO ? (C64 ? 3 : 4) : 2;
  const int ntiles = (cend - cbeg) * TPC;
  const int sbase = (slice % NSL) * SW;           // first state column of the slice
  const int g32 = warp < NCW ? (warp >> 2) : 0;   // compute threads: 32-column group in the slice
  const int col0 = sbase + 32 * g32;              // first state column of this thread's values
  // The recompute mode stages its exported h and Delta slices in the last slot
  // (8 KiB each, double-buffered, 64-byte swizzle; a store warp writes them
  // out) and streams its 2 tiles per chunk through a 5-slot ring.  The output
  // mode needs all 6 slots for its 4 tiles per chunk and stores O rows
  // directly (measured faster than staging it at 5 slots); the fold pass
  // stores nothing per chunk.
  constexpr bool staged = STAGED;
  constexpr int nring = STAGED ? NSLOT - 1 : NSLOT;  // compile-time: the ring index is on the issue path
  unsigned char* stage = sm.slot[NSLOT - 1];
  if (cbeg >= cend) return;
  if (partA && a.pairA == nullptr) return;  // fold without the A output: B columns only
  auto rows_of = [&](int c) { return min(CC, a.T - c * CC); };
  // tile sequence of a chunk: w, Q, K, P (with output) or w, K
  auto tile_of = [&](int kind) { return withO ? kind : (kind == 0 ? 0 : 1); };  // kind: 0 w, 1 Q, 2 K, 3 P
  // first workspace row (w, u, P) of chunk c: 128-row tiles, two 64-token chunks to a tile
  auto ws_row = [&](int c) { return bh * a.NT * CH + (long)c * CC; };

  if (tid == 0) {
    for (int k = 0; k < NSLOT; ++k) {
      tc::mbar_init(&sm.full[k], 1);
      tc::mbar_init(&sm.empty[k], 1);
    }
    tc::mbar_init(&sm.barX, 1);
    tc::mbar_init(&sm.barO1, 1);
    tc::mbar_init(&sm.barH, 1);
    tc::mbar_init(&sm.barO2, 1);
    tc::mbar_init(&sm.barDg, NCT);
    tc::mbar_init(&sm.barD, NCT);
    tc::mbar_init(&sm.barHt, NCT);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&sm.sfull[k], NCT);
      tc::mbar_init(&sm.sempty[k], 1);
    }
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::alloc(&sm.tmem, Cfg::TMEM_COLS);
  bool ok = true;
  pdl_wait();  // before any load of what earlier kernels wrote, and any store
  pdl_release();

  // state row r = tid (compute threads), columns col0..col0+31
  const int r = 32 * (warp & 3) + lane;
  // with 64-token chunks rows 0-63 form Delta and rows 64-127 the output, both
  // of token r & 63 (warp-uniform); every thread keeps state row r
  const bool dRow = !C64 || r < 64;
  const int tr = C64 ? (r & 63) : r;
  float h[32];
  float gnext = 0.f, part = 0.f;
  float gam_r = 0.f, ef_r = 0.f, gC = 0.f;
  auto load_g = [&](int c) {
    return (c < cend && tr < rows_of(c)) ? act_g(a.g[((long)b * a.T + (long)c * CC + tr) * a.Hv + j], a.gate_logits)
                                         : 0.f;
  };
  // row r of this slice of u for chunk c, loaded a chunk ahead into registers
  uint4 un[4];
  auto load_u = [&](int c) {
    if (partA || c >= cend || !dRow) return;
    const bf16* src = a.U + (ws_row(c) + r) * HD + col0;
#pragma unroll
    for (int q = 0; q < 4; ++q) un[q] = *reinterpret_cast<const uint4*>(src + 8 * q);
  };
  // gate totals of chunk index i (from the segment start) go to gsum[i & 1]:
  // a warp may post the totals of chunk i + 1 while another still reads those of i
  auto scan_part = [&](float gv, int i) {  // warp-inclusive scan; warp totals to smem
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, gv, off);
      if (lane >= off) gv += o;
    }
    if (lane == 31) sm.gsum[i & 1][warp & 3] = gv;  // both column groups post the same totals
    return gv;
  };
  // raw K and Q rows (a.nrm): this row's 1/||k|| and 1/||q|| in chunk c, which
  // scale ef (the state update reads K) and gamma (the output reads Q)
  float nk_next = 1.f, nq_next = 1.f;
  auto load_n = [&](int c, float& nk, float& nq) {
    nk = nq = 1.f;
    if (a.nrm && c < cend) {
      const int t = C64 ? (c >> 1) : c, o = C64 ? 64 * (c & 1) + tr : r;  // tile, row in it
      const float* nb = a.nrm + ((((long)b * a.Hk + kh) * a.NT + t) << 8);
      nk = nb[o];
      nq = nb[CH + o];
    }
  };
  // after a barrier over the compute threads: gamma_r, ef_r and gamma_C of chunk index i
  // (64-token chunks: lane quarters 0-1 and 2-3 each scan the chunk's 64 gates)
  auto finish_gates = [&](float p, int i, float& gm, float& ef, float& gc) {
    float off = 0.f, tot = 0.f;
    if (C64) {
      const int q0 = warp & 2;
      off = (warp & 1) ? sm.gsum[i & 1][q0] : 0.f;
      tot = sm.gsum[i & 1][q0] + sm.gsum[i & 1][q0 + 1];
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float s = sm.gsum[i & 1][w];
        off += (w < (warp & 3)) ? s : 0.f;
        tot += s;
      }
    }
    const float G = p + off;
    gm = expf(G) * nq_next;  // the norms of chunk index i were loaded a chunk ahead
    ef = expf(tot - G) * nk_next;
    gc = expf(tot);
  };
  if (warp < NCW) {
    if (FOLD) {
#pragma unroll
      for (int n = 0; n < 32; ++n) h[n] = (partA && r == col0 + n) ? 1.f : 0.f;
    } else {
      const float* hs = a.hstart ? a.hstart + bh * a.hstart_bh_stride + seg * a.hstart_seg_stride : nullptr;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hs) x = *reinterpret_cast<const float4*>(hs + (long)r * HD + col0 + 4 * q);
        h[4 * q] = x.x;
        h[4 * q + 1] = x.y;
        h[4 * q + 2] = x.z;
        h[4 * q + 3] = x.w;
      }
    }
    write_bt_column<SW>(sm.Ht[0], r, 32 * g32, h);
    load_u(cbeg);
    part = scan_part(load_g(cbeg), 0);
    gnext = load_g(cbeg + 1);
    load_n(cbeg, nk_next, nq_next);
  }
  tc::fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // TMEM columns: X = w h at 0, H' at SW, P Delta at 3 SW; Q h alternates between
  // 2 SW and 4 SW (it is read after the next chunk's Q h may have been issued)
  const uint32_t tmem = sm.tmem;
  constexpr uint32_t C_H = SW, C_O2 = 3 * SW;
  auto o1_col = [](int ci) { return (ci & 1) ? 4u * SW : 2u * SW; };

  auto issue = [&](int i) {  // TMA request of tile i into slot i % nring
    const int c = cbeg + i / TPC, t = i % TPC;
    if (C64) {  // 64-row boxes: [w; Q] (or w), K, P into rows 64-127 of the first half
      const int row0 = (int)ws_row(c);
      unsigned char* dst = sm.slot[i % nring];
      uint64_t* bar = &sm.full[i % nring];
      if (t == 0) {
        tc::arrive_expect_tx(bar, withO ? TILE_BYTES : TILE_BYTES / 2);
        tc::tma_load_2d(dst, &mp.W, 0, row0, bar);
        tc::tma_load_2d(dst + TILE_BYTES / 2, &mp.W, 64, row0, bar);
        if (withO) {
          tc::tma_load_4d(dst + TILE_BYTES / 4, &mp.q, 0, kh, c * CC, b, bar);
          tc::tma_load_4d(dst + TILE_BYTES / 2 + TILE_BYTES / 4, &mp.q, 64, kh, c * CC, b, bar);
        }
      } else if (t == 1) {
        tc::arrive_expect_tx(bar, TILE_BYTES / 2);
        tc::tma_load_4d(dst, &mp.k, 0, kh, c * CC, b, bar);
        tc::tma_load_4d(dst + TILE_BYTES / 2, &mp.k, 64, kh, c * CC, b, bar);
      } else {
        tc::arrive_expect_tx(bar, TILE_BYTES / 4);
        tc::tma_load_2d(dst + TILE_BYTES / 4, &mp.P, 64 * (c & 1), row0, bar);
      }
      return;
    }
    const int kind = withO ? t : (t == 0 ? 0 : 2);
    const long cid = bh * a.NC + c;
    unsigned char* dst = sm.slot[i % nring];
    uint64_t* bar = &sm.full[i % nring];
    tc::arrive_expect_tx(bar, TILE_BYTES);
    if (kind == 0 || kind == 3) {
      const CUtensorMap* m = (kind == 0) ? &mp.W : &mp.P;
      tc::tma_load_2d(dst, m, 0, (int)(cid * CH), bar);
      tc::tma_load_2d(dst + TILE_BYTES / 2, m, 64, (int)(cid * CH), bar);
    } else {
      const CUtensorMap* m = (kind == 1) ? &mp.q : &mp.k;
      tc::tma_load_4d(dst, m, 0, kh, c * CH, b, bar);
      tc::tma_load_4d(dst + TILE_BYTES / 2, m, 64, kh, c * CH, b, bar);
    }
  };

  if (warp == NCW + 2 && withO) {
    // ======================================================= output products
    // Q h(c) once w h(c) has completed (the chain's product goes first) and
    // P Delta(c) once Delta^T is written, issued from this warp so that their
    // issue never holds the chain's issuer.  The compute threads wait for
    // P Delta(c) (which covers Q h(c), issued before it from this thread)
    // before they overwrite the images or the output columns these read.
    if (lane == 0) {
      auto wait_tile = [&](int i) { ok = ok && tc::mbar_wait_sleep(&sm.full[i % nring], (i / nring) & 1); };
      auto slot_of = [&](int i) { return smem_u32(sm.slot[i % nring]); };
      auto release = [&](int i) { tc::commit(&sm.empty[i % nring]); };
      for (int c = cbeg; c < cend; ++c) {
        const int ci = c - cbeg;
        const uint32_t par = (uint32_t)(ci & 1);
        if (C64) {  // Q h came with w h; P Delta alone, K = 64
          const int iP = ci * TPC + 2;
          wait_tile(iP);  // (the tile first: it is in long before Delta)
          ok = ok && tc::mbar_wait_sleep(&sm.barD, par);  // Delta^T written
          tc::fence_after();
          tc::gemm_k128<4>(tmem + C_O2, slot_of(iP), smem_u32(sm.Dt), SW, false);
          tc::commit(&sm.barO2);
          release(iP);
          continue;
        }
        const int iQ = ci * TPC + 1, iP = ci * TPC + 3;
        wait_tile(iQ);  // (the tile first: it is in long before w h)
        ok = ok && tc::mbar_wait_sleep(&sm.barX, par);  // w h(c) done: h(c) is in Ht[ci & 1]
        tc::fence_after();
        tc::gemm_k128(tmem + o1_col(ci), slot_of(iQ), smem_u32(sm.Ht[ci & 1]), SW, false);
        tc::commit(&sm.barO1);
        release(iQ);
        wait_tile(iP);
        ok = ok && tc::mbar_wait_sleep(&sm.barD, par);  // Delta^T written
        tc::fence_after();
        tc::gemm_k128(tmem + C_O2, slot_of(iP), smem_u32(sm.Dt), SW, false);
        tc::commit(&sm.barO2);
        release(iP);
      }
    }
  } else if (warp == (withO ? NCW + 3 : NCW + 2)) {
    // ============================================================ TMA stores
    // (with output, the block has a fourth extra warp for them)
    // The h and Delta slices staged for chunk index i leave by TMA stores once
    // the compute threads have signalled them; when the stores have read the
    // buffers they are handed back.  A store request can block its thread, so
    // it never runs on a compute or issuing thread.
    if (staged && lane == 0) {
      for (int c = cbeg; c < cend; ++c) {
        const int ci = c - cbeg;
        const int set = ci % NSTAGE, use = ci / NSTAGE;
        ok = ok && tc::mbar_wait_sleep(&sm.sfull[set], (uint32_t)(use & 1));
        if (a.states) tc::tma_store_2d(&mp.St, sbase, (int)((bh * a.NC + c) * HD), stage + set * 2 * SLICE);
        if (a.delta) tc::tma_store_2d(&mp.De, sbase, (int)((bh * a.NC + c) * CH), stage + set * 2 * SLICE + SLICE);
        tc::bulk_commit();
        tc::bulk_wait_read();
        arrive(&sm.sempty[set]);
      }
      tc::bulk_wait();  // every store has completed before the block exits
    }
  } else if (warp == NCW + 1) {
    // ========================================================== TMA producer
    // Tile i goes into slot i % nring once the product that read tile
    // i - nring has completed (signalled on that slot's empty barrier).
    if (lane == 0) {
      for (int i = 0; i < ntiles; ++i) {
        if (i >= nring) ok = ok && tc::mbar_wait_sleep(&sm.empty[i % nring], (uint32_t)((i / nring - 1) & 1));
        if (!ok) break;  // a wait gave up: request nothing more (the CTA ends soon)
        issue(i);
      }
    }
  } else if (warp == NCW) {
    // ================================================================ MMA issuer
    // Chain products first: w h(c) as soon as the state image is written, then
    // K^T (ef Delta) as soon as Delta is; Q h(c) and P Delta fill the gaps.  An
    // MMA issue returns about when the tensor core has taken it, so the order
    // of issue is the order of execution.  After each product its tile slot is
    // released to the producer by a commit to the slot's empty barrier.
    if (lane == 0) {
      auto wait_tile = [&](int i) { ok = ok && tc::mbar_wait_sleep(&sm.full[i % nring], (i / nring) & 1); };
      auto slot_of = [&](int i) { return smem_u32(sm.slot[i % nring]); };
      auto release = [&](int i) { tc::commit(&sm.empty[i % nring]); };
      for (int c = cbeg; c < cend; ++c) {
        const int ci = c - cbeg;
        const uint32_t par = (uint32_t)(ci & 1);
        const int t0 = ci * TPC;
        const int iW = t0, iQ = t0 + 1, iK = t0 + (C64 ? 1 : tile_of(2)), iP = t0 + 3;
        const uint32_t ht = smem_u32(sm.Ht[ci & 1]);
        // (each tile is waited for before the compute threads' signal: the tiles
        // are in long before it, so the product issues as soon as the signal comes)
        wait_tile(iW);
        if (ci > 0) ok = ok && tc::mbar_wait_sleep(&sm.barHt, par ^ 1);  // state image of chunk c
        tc::fence_after();
        tc::gemm_k128(tmem + 0, slot_of(iW), ht, SW, false);
        tc::commit(&sm.barX);
        release(iW);
        wait_tile(iK);
        ok = ok && tc::mbar_wait_sleep(&sm.barDg, par);  // (ef Delta)^T written
        tc::fence_after();
        if (C64)
          tc::gemm_amn_k128<4>(tmem + C_H, slot_of(iK), smem_u32(sm.Dgt), SW, false);
        else
          tc::gemm_amn_k128(tmem + C_H, slot_of(iK), smem_u32(sm.Dgt), SW, false);
        tc::commit(&sm.barH);
        release(iK);
        (void)iQ;
        (void)iP;
      }
    }
  } else if (warp < NCW) {
    // ========================================================== compute threads
    finish_gates(part, 0, gam_r, ef_r, gC);
    load_n(cbeg + 1, nk_next, nq_next);
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32u * g32;  // lanes of this warp, its columns
    for (int c = cbeg; c < cend; ++c) {
      const int ci = c - cbeg;
      const uint32_t par = (uint32_t)(ci & 1);
      // staging set ci % NSTAGE (h, Delta) was last read by the stores of chunk ci - NSTAGE
      const int set = ci % NSTAGE, use = ci / NSTAGE;
      if (staged && use >= 1) ok = ok && tc::mbar_wait_sleep(&sm.sempty[set], (uint32_t)((use - 1) & 1));
      if (!FOLD && a.states) stage_row<SW>(stage + set * 2 * SLICE, r, g32, h);

      // ---- Delta = u - X -------------------------------------------------------
      ok = ok && tc::mbar_wait_sleep(&sm.barX, par);
      tc::fence_after();
      float x[32];  // (64-token chunks, rows 64-127: Q h, kept for the output)
      tc::ld32(tl + 0, x);
      if (!dRow) {
      } else if (!partA) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w4 = un[q];
          const float2 f0 = unpack_bf16(w4.x), f1 = unpack_bf16(w4.y), f2 = unpack_bf16(w4.z),
                       f3 = unpack_bf16(w4.w);
          x[8 * q] = f0.x - x[8 * q];
          x[8 * q + 1] = f0.y - x[8 * q + 1];
          x[8 * q + 2] = f1.x - x[8 * q + 2];
          x[8 * q + 3] = f1.y - x[8 * q + 3];
          x[8 * q + 4] = f2.x - x[8 * q + 4];
          x[8 * q + 5] = f2.y - x[8 * q + 5];
          x[8 * q + 6] = f3.x - x[8 * q + 6];
          x[8 * q + 7] = f3.y - x[8 * q + 7];
        }
      } else {
#pragma unroll
        for (int n = 0; n < 32; ++n) x[n] = -x[n];
      }
      if (dRow) {
        float xg[32];
#pragma unroll
        for (int n = 0; n < 32; ++n) xg[n] = x[n] * ef_r;
        write_bt_column<SW>(sm.Dgt, r, 32 * g32, xg);  // operand of the state update: first
      }
      tc::fence_proxy_async();
      tc::fence_before();
      arrive(&sm.barDg);
      load_u(c + 1);
      if (withO) {
        // (every compute thread arrives: P Delta(c) then also waits for the
        // output rows' reads of P Delta(c - 1))
        if (dRow) write_bt_column<SW>(sm.Dt, r, 32 * g32, x);
        tc::fence_proxy_async();
        tc::fence_before();
        arrive(&sm.barD);
      }
      if (!FOLD && a.delta) stage_row<SW>(stage + set * 2 * SLICE + SLICE, r, g32, x);
      if (staged) {  // h and Delta of this chunk are staged
        tc::fence_proxy_async();
        arrive(&sm.sfull[set]);
      }

      // ---- gates of chunk c + 1, while K^T (ef Delta) runs ----------------------------
      float gam_n, ef_n, gC_n;
      part = scan_part(gnext, ci + 1);
      gnext = load_g(c + 2);
      asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
      finish_gates(part, ci + 1, gam_n, ef_n, gC_n);
      load_n(c + 2, nk_next, nq_next);

      // ---- h' = gamma_C h + H' ---------------------------------------------------
      ok = ok && tc::mbar_wait_sleep(&sm.barH, par);
      tc::fence_after();
      float hh[32];
      tc::ld32(tl + C_H, hh);
#pragma unroll
      for (int n = 0; n < 32; ++n) h[n] = gC * h[n] + hh[n];
      // the other image buffer held h of the previous chunk, whose readers have completed
      write_bt_column<SW>(sm.Ht[(ci + 1) & 1], r, 32 * g32, h);
      tc::fence_proxy_async();
      tc::fence_before();
      arrive(&sm.barHt);
      if (withO && C64) {  // rows 64-127: O = gamma (Q h) + P Delta
        ok = ok && tc::mbar_wait_sleep(&sm.barO2, par);
        tc::fence_after();
        if (!dRow) {
          float o2[32];
          tc::ld32(tl + C_O2, o2);
          if (tr < rows_of(c)) {
#pragma unroll
            for (int n = 0; n < 32; ++n) o2[n] = gam_r * x[n] + o2[n];
            store_row_bf16(a.o + (((long)b * a.T + (long)c * CC + tr) * a.Hv + j) * HD + col0, o2);
          }
        }
      } else if (withO) {  // output epilogue overlaps the next chunk's first product
        ok = ok && tc::mbar_wait_sleep(&sm.barO2, par);  // covers Q h as well
        tc::fence_after();
        float o1[32], o2[32];
        tc::ld32(tl + o1_col(ci), o1);
        tc::ld32(tl + C_O2, o2);
        if (r < rows_of(c)) {
#pragma unroll
          for (int n = 0; n < 32; ++n) o1[n] = gam_r * o1[n] + o2[n];
          store_row_bf16(a.o + (((long)b * a.T + (long)c * CH + r) * a.Hv + j) * HD + col0, o1);
        }
      }
      gam_r = gam_n;
      ef_r = ef_n;
      gC = gC_n;
    }
    if (FOLD) {
      float* dst = (partA ? a.pairA : a.pairB) + ((bh * a.S + seg) * HD + r) * HD + col0;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    } else if (a.hT && seg == a.S - 1) {
      float* dst = a.hT + (bh * HD + r) * HD + col0;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    }
  }
  if (!ok && a.status) atomicOr(a.status, 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, Cfg::TMEM_COLS);
}

}  // namespace walkf
}  // namespace gdn
