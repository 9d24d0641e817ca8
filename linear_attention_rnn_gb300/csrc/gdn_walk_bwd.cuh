// gdn_walk_bwd.cuh -- reverse walk of the state cotangent over the chunks of a segment
// (device body; the kernels that run it are in gdn_walk_bwd.cu and gdn_walk_pair.cu).
//
// The backward "walks the chunks in reverse" ("Fuse the Gated Delta Net
// inter-chunk scan into a Pallas TPU kernel", section "Changes").  With dh' the
// cotangent of the state leaving chunk c, the chunk forward
//     Delta = u - w h,  O = diag(gamma) Q h + P Delta,  h' = gamma_C h + k_g^T Delta
// gives
//     Y = dDelta = diag(ef) K dh' + P^T dO
//     dh = gamma_C dh' + Q^T diag(gamma) dO - w^T Y,
// an affine map of dh' with matrix A_c^T, so it segments exactly like the
// forward (the transposed maps compose in reverse order).
//
// One CTA walks a slice of SW = 32 or 64 columns of dh (columns are
// independent).  Compute thread (r, g) owns row r, columns 32 g .. 32 g + 31
// of the slice in fp32 registers, and those columns of TMEM lane r in every
// product.  A product costs about its A-tile read whatever N is, so a 64-column
// slice does twice the work per product for about 10% more time and leaves
// half the SMs free.  Per chunk the tcgen05 products (M = 128, N = SW, K = 128)
//     K dh'            (A = K, K-major)
//     P^T dO           (A = the P tile read MN-major)
//     Q^T (gamma dO)   (A = the Q tile read MN-major), then += w^T (-Y) on top
//                      (A = the w tile read MN-major)
// take B operands written column by column by the compute threads (dh'^T,
// dO^T, (gamma dO)^T, (-Y)^T, SW x 128 bf16, 128-byte-swizzled K-major); on
// 32-column slices P^T dO reads the chunk's dO slice instead, as TMA stored it.  The
// two dO products do not depend on dh', so they run ahead of the chain
// dh' -> Y -> dh.  A fifth warp issues the MMAs once their operands are
// signalled ready; a sixth issues the TMA loads of the chunk tiles (P, Q, K, w
// in the order consumed) into a ring of 32 KiB slots, refilling each as
// soon as the MMA that read it completes.  With SPLIT (the kernels that run
// this walk alone) an eighth warp issues the two dO products, so that their
// issue never holds the chain's issuer; the chain's issuer then waits for
// Q^T (gamma dO) to complete before it accumulates w^T (-Y) onto it.  The
// compute threads form the dO images from each chunk's dO rows.  On 32-column
// slices those rows arrive by TMA into one of two slice buffers (the store warp
// requests each chunk's slice once the images of the chunk before are written),
// so the compute threads issue no global loads: an mbarrier arrive, a release,
// would wait for them.  There P^T dO reads the slice directly (MN-major, 64-byte
// swizzle) and only (gamma dO)^T is written as an image.
// Every wait is bounded; one that gives up sets bit 0 of the status word.
//
// Modes:
//   WALK (fold = 0): from the cotangent leaving the segment, store for every
//     chunk the bf16 cotangent of the state leaving it and dDelta; segment 0
//     writes dh0 (the cotangent of the initial state).
//   FOLD (fold = 1): push [Abar | Bbar] from [I | 0] backwards through the
//     segment's chunks; the Abar columns take no dO terms.  The result maps
//     the cotangent leaving the segment to the one entering it:
//     dh_in = Abar dh_out + Bbar.
#pragma once
#include "gdn_kernels.cuh"
#include "gdn_tc05.cuh"

namespace gdn {
namespace walkb {

constexpr uint32_t TILE_BYTES = CH * HD * 2;  // 32 KiB

// Layout per slice width SW (state columns per CTA: 32 or 64)
template <int SW>
struct BwdCfg {
  static constexpr int NCT = 4 * SW;               // compute threads: 4 lane quarters x SW / 32 column groups
  static constexpr int NCW = NCT / 32;             // compute warps
  static constexpr int NT = NCT + 96;              // + MMA issuer, TMA producer and TMA store warps
  static constexpr int NRING = SW == 32 ? 5 : 4;   // tile ring
  static constexpr int NSTAGE = 1;                 // staging sets of the stored dh' and dDelta slices
  // SW 32: each chunk's dO slice arrives by TMA into shared memory (dOt), so
  // the compute threads issue no global loads: their every arrive (a release)
  // would wait for those loads to return.
  static constexpr bool DOTMA = SW == 32;
  static constexpr uint32_t BT = SW * HD * 2;      // a [SW x 128] B-operand image
  static constexpr uint32_t SLICE = CH * SW * 2;   // a [128 x SW] staged slice
  static constexpr uint32_t TMEM_COLS = 4 * SW;    // K dh', P^T dO, Q^T (gamma dO) - w^T Y twice
};

template <int SW>
struct WalkBwdSmem {
  using C = BwdCfg<SW>;
  unsigned char slot[C::NRING][TILE_BYTES];
  unsigned char stage[C::NSTAGE][2][C::SLICE];  // [set][dh', dDelta]; SW 32: 64-byte, SW 64: 128-byte swizzle
  unsigned char Xt[C::BT];   // dh'^T
  unsigned char Yt[C::BT];   // (-Y)^T
  unsigned char Ot[C::BT];   // dO^T (this slice); DOTMA: the second dO-slice buffer
  unsigned char Ogt[C::BT];  // (diag(gamma) dO)^T
  unsigned char dOt[C::DOTMA ? C::SLICE : 16];  // DOTMA: dO slice [128 x 32] of even chunk indices, 64-byte swizzle
  float gsum[2][4];
  uint64_t full[C::NRING], empty[C::NRING];
  uint64_t barO, barXt, barYt, barQ, barY, barH;  // barY: K dh' and P^T dO complete
  uint64_t sfull[C::NSTAGE], sempty[C::NSTAGE];  // staging set: written by the compute threads / read by its stores
  uint64_t barDO;  // DOTMA: dOt loaded
  uint32_t tmem;
};

// Column k of a [SW x 128] K-major SW128 B image: rows n0 .. n0 + 31 from 32 fp32 values.
template <int SW>
__device__ __forceinline__ void write_bt_column(unsigned char* tile, int k, int n0, const float (&v)[32]) {
#pragma unroll
  for (int n = 0; n < 32; ++n)
    *reinterpret_cast<bf16*>(tile + tc::sw128(n0 + n, k, SW)) = __float2bfloat16_rn(v[n]);
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
__device__ __forceinline__ void store_row_f32(float* dst, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The walk of CTA (slice, seg, bhi) with BwdCfg<SW>::NT threads; `base` is the
// 1024-byte-aligned dynamic shared memory (sizeof(WalkBwdSmem<SW>) bytes).
template <bool FOLD, int SW, bool SPLIT = false>
__device__ __forceinline__ void walk(const WalkBwdArgs& a, const WalkBwdMaps& mp, unsigned char* base, int slice,
                                     int seg, int bhi) {
  using Cfg = BwdCfg<SW>;
  constexpr int NCT = Cfg::NCT, NCW = Cfg::NCW, NRING = Cfg::NRING, NSTAGE = Cfg::NSTAGE;
  constexpr bool DOTMA = Cfg::DOTMA;
  constexpr int NSL = HD / SW;  // slices per state
  // TMEM columns: K dh' at 0, P^T dO at SW; Q^T (gamma dO) - w^T Y alternates 2 SW / 3 SW
  constexpr uint32_t C_Y = 0, C_P = SW;
  auto c_q = [](int ci) { return (ci & 1) ? 3u * SW : 2u * SW; };
  WalkBwdSmem<SW>& sm = *reinterpret_cast<WalkBwdSmem<SW>*>(base);
  const int b = bhi / a.Hv, j = bhi % a.Hv, kh = j / (a.Hv / a.Hk);
  const long bh = bhi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cbeg = (int)((long)seg * a.NC / a.S), cend = (int)((long)(seg + 1) * a.NC / a.S);
  const bool partA = FOLD && slice < NSL;  // Abar columns: no dO terms
  const bool withO = !partA;
  const int TPC = withO ? 4 : 2;  // tiles per chunk: P, Q, K, w (or K, w)
  const int n = cend - cbeg;
  const int ntiles = n * TPC;
  const int sbase = (slice % NSL) * SW;           // first state column of the slice
  const int g32 = warp < NCW ? (warp >> 2) : 0;   // compute threads: 32-column group in the slice
  const int col0 = sbase + 32 * g32;              // first state column of this thread's values
  if (n <= 0) return;
  auto chunk_of = [&](int ci) { return cend - 1 - ci; };  // walk order
  auto rows_of = [&](int c) { return min(CH, a.T - c * CH); };

  if (tid == 0) {
    for (int k = 0; k < NRING; ++k) {
      tc::mbar_init(&sm.full[k], 1);
      tc::mbar_init(&sm.empty[k], 1);
    }
    tc::mbar_init(&sm.barO, NCT);
    tc::mbar_init(&sm.barXt, NCT);
    tc::mbar_init(&sm.barYt, NCT);
    tc::mbar_init(&sm.barQ, 1);
    // SPLIT: the chain's issuer (K dh') and the dO products' issuer (P^T dO) both
    // commit to barY; otherwise the chain's issuer issues P^T dO before K dh'
    tc::mbar_init(&sm.barY, (SPLIT && withO) ? 2 : 1);
    tc::mbar_init(&sm.barH, 1);
    tc::mbar_init(&sm.barDO, 1);
    for (int k = 0; k < NSTAGE; ++k) {
      tc::mbar_init(&sm.sfull[k], NCT);
      tc::mbar_init(&sm.sempty[k], 1);
    }
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::alloc(&sm.tmem, Cfg::TMEM_COLS);
  bool ok = true;
  pdl_wait();  // before any load of what earlier kernels wrote, and any store
  pdl_release();

  const int r = 32 * (warp & 3) + lane;  // compute threads: row r of the state slice / of the chunk
  float x[32];
  float gnext = 0.f, part = 0.f;  // gnext: the raw gate entry of row r of a later chunk
  float gam_r = 0.f, ef_r = 0.f, gC = 0.f;
  uint4 don[4];  // dO row r of the first chunk's images (this thread's 32 columns)
  auto has_row = [&](int ci) { return ci < n && r < rows_of(chunk_of(ci)); };
  // The loads land in their registers untouched (ld_pred_*): the raw gate is
  // activated, and the dO row unpacked, where they are used, long after the load.
  auto load_g = [&](int ci) {
    float v = 0.f;
    const bool in = has_row(ci);
    ld_pred_f32(v, a.g + ((long)b * a.T + (long)chunk_of(in ? ci : 0) * CH + (in ? r : 0)) * a.Hv + j, in);
    return v;
  };
  auto gate_of = [&](float raw, int ci) { return has_row(ci) ? act_g(raw, a.gate_logits) : 0.f; };
  auto load_do = [&](int ci, uint4 (&dst)[4]) {
    const bool in = withO && has_row(ci);
    const bf16* src = a.dO + (((long)b * a.T + (long)chunk_of(in ? ci : 0) * CH + (in ? r : 0)) * a.Hv + j) * HD + col0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dst[q] = make_uint4(0u, 0u, 0u, 0u);
      ld_pred_v4(dst[q], src + 8 * q, in);
    }
  };
  // DOTMA: the dO slice of chunk index i lies in dO_slice(i), where P^T dO reads it
  // directly (MN-major); only (gamma dO)^T is written as an image
  static_assert(!DOTMA || (SPLIT && Cfg::SLICE == Cfg::BT), "the slice buffers take the dO^T image's place");
  auto dO_slice = [&](int i) { return (i & 1) ? sm.Ot : sm.dOt; };
  // dO^T (unless DOTMA) and (gamma dO)^T images of the chunk whose dO rows are in dn
  auto write_do_images = [&](const uint4 (&dn)[4]) {
    float d[32], dg[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w4[4] = {dn[q].x, dn[q].y, dn[q].z, dn[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16(w4[e]);
        d[8 * q + 2 * e] = f.x;
        d[8 * q + 2 * e + 1] = f.y;
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) dg[i] = gam_r * d[i];
    if (!DOTMA) write_bt_column<SW>(sm.Ot, r, 32 * g32, d);
    write_bt_column<SW>(sm.Ogt, r, 32 * g32, dg);
  };
  auto scan_part = [&](float gv, int i) {  // warp-inclusive scan; warp totals to gsum[i & 1]
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, gv, off);
      if (lane >= off) gv += o;
    }
    if (lane == 31) sm.gsum[i & 1][warp & 3] = gv;  // both column groups post the same totals
    return gv;
  };
  auto finish_gates = [&](float p, int i) {  // after a barrier over the compute threads
    float off = 0.f, tot = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float s = sm.gsum[i & 1][w];
      off += (w < (warp & 3)) ? s : 0.f;
      tot += s;
    }
    const float G = p + off;
    gam_r = expf(G);
    ef_r = expf(tot - G);
    gC = expf(tot);
  };
  if (warp < NCW) {
    if (FOLD) {
#pragma unroll
      for (int q = 0; q < 32; ++q) x[q] = (partA && r == col0 + q) ? 1.f : 0.f;
    } else {
      const float* hs = a.hstart ? a.hstart + bh * a.hstart_bh_stride + seg * a.hstart_seg_stride : nullptr;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hs) v = *reinterpret_cast<const float4*>(hs + (long)r * HD + col0 + 4 * q);
        x[4 * q] = v.x;
        x[4 * q + 1] = v.y;
        x[4 * q + 2] = v.z;
        x[4 * q + 3] = v.w;
      }
    }
    write_bt_column<SW>(sm.Xt, r, 32 * g32, x);
    part = scan_part(gate_of(load_g(0), 0), 0);
    gnext = load_g(1);
    load_do(0, don);
  }
  tc::fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem;

  auto issue = [&](int i) {  // TMA request of tile i into slot i % NRING
    const int ci = i / TPC, t = i % TPC;
    const int c = chunk_of(ci);
    const int kind = withO ? t : (t == 0 ? 2 : 3);  // 0 P, 1 Q, 2 K, 3 w
    const long cid = bh * a.NC + c;
    unsigned char* dst = sm.slot[i % NRING];
    uint64_t* bar = &sm.full[i % NRING];
    tc::arrive_expect_tx(bar, TILE_BYTES);
    if (kind == 0 || kind == 3) {
      const CUtensorMap* m = (kind == 0) ? &mp.P : &mp.W;
      tc::tma_load_2d(dst, m, 0, (int)(cid * CH), bar);
      tc::tma_load_2d(dst + TILE_BYTES / 2, m, 64, (int)(cid * CH), bar);
    } else {
      const CUtensorMap* m = (kind == 1) ? &mp.q : &mp.k;
      tc::tma_load_4d(dst, m, 0, kh, c * CH, b, bar);
      tc::tma_load_4d(dst + TILE_BYTES / 2, m, 64, kh, c * CH, b, bar);
    }
  };

  if (SPLIT && warp == NCW + 3) {
    // ===================================================== dO products' issuer
    // P^T dO and Q^T (gamma dO) of each chunk once its dO images are written
    // (they were written after both products of the chunk before had read them)
    if (lane == 0 && withO) {
      for (int ci = 0; ci < n; ++ci) {
        const int t0 = ci * TPC;
        ok = ok && tc::mbar_wait_sleep(&sm.full[t0 % NRING], (t0 / NRING) & 1);  // (tile first)
        ok = ok && tc::mbar_wait_sleep(&sm.barO, (uint32_t)(ci & 1));
        tc::fence_after();
        if (DOTMA)
          tc::gemm_amn_bmn64_k128(tmem + C_P, smem_u32(sm.slot[t0 % NRING]), smem_u32(dO_slice(ci)));
        else
          tc::gemm_amn_k128(tmem + C_P, smem_u32(sm.slot[t0 % NRING]), smem_u32(sm.Ot), SW, false);
        tc::commit(&sm.barY);  // (barY's second arrival of the chunk)
        tc::commit(&sm.empty[t0 % NRING]);
        const int iQ = t0 + 1;
        ok = ok && tc::mbar_wait_sleep(&sm.full[iQ % NRING], (iQ / NRING) & 1);
        tc::fence_after();
        tc::gemm_amn_k128(tmem + c_q(ci), smem_u32(sm.slot[iQ % NRING]), smem_u32(sm.Ogt), SW, false);
        tc::commit(&sm.barQ);
        tc::commit(&sm.empty[iQ % NRING]);
      }
    }
  } else if (warp == NCW + 2) {
    // ============================================================ TMA stores
    // The staged dh' and dDelta slices of each chunk leave by TMA stores once the
    // compute threads have signalled them; when the stores have read the buffers
    // they are handed back.  A store request can block its thread.  DOTMA: this
    // thread also loads each chunk's dO slice into dOt, once the compute
    // threads have written the images of the chunk before from it (barO).
    const bool stores = !FOLD && (a.dstates || a.ddelta);
    const bool dol = DOTMA && withO;
    auto load_slice = [&](int ci) {  // dO slice of chunk index ci (rows past T read as zero)
      tc::arrive_expect_tx(&sm.barDO, Cfg::SLICE);
      tc::tma_load_4d(dO_slice(ci), &mp.dO, col0, j, chunk_of(ci) * CH, b, &sm.barDO);
    };
    if (lane == 0 && (stores || dol)) {
      // barO's phases are waited for in order, from phase 0 (the images of chunk
      // index 0, from plain loads), each while barO is in it or just past it: a
      // parity wait for the phase after the current one would pass at once, one
      // for a phase two back would not pass.  Its phase ci + 1 needs the slice
      // of chunk index ci + 1, loaded only after the wait for phase ci.
      if (dol && n > 1) {
        ok = ok && tc::mbar_wait_sleep(&sm.barO, 0u);
        if (ok) load_slice(1);
      }
      for (int ci = 0; ci < n; ++ci) {
        if (stores) {
          const int c = chunk_of(ci);
          const int set = ci % NSTAGE, use = ci / NSTAGE;
          ok = ok && tc::mbar_wait_sleep(&sm.sfull[set], (uint32_t)(use & 1));
          if (a.dstates) tc::tma_store_2d(&mp.Ds, sbase, (int)((bh * a.NC + c) * HD), sm.stage[set][0]);
          if (a.ddelta) tc::tma_store_2d(&mp.Dd, sbase, (int)((bh * a.NC + c) * CH), sm.stage[set][1]);
          tc::bulk_commit();
          tc::bulk_wait_read();
          arrive(&sm.sempty[set]);
        }
        if (dol && ci + 2 < n) {  // the images of chunk index ci + 1 are written
          ok = ok && tc::mbar_wait_sleep(&sm.barO, (uint32_t)((ci + 1) & 1));
          if (ok) load_slice(ci + 2);
        }
      }
      if (stores) tc::bulk_wait();  // every store has completed before the block exits
    }
  } else if (warp == NCW + 1) {
    // ========================================================== TMA producer
    if (lane == 0) {
      for (int i = 0; i < ntiles; ++i) {
        if (i >= NRING) ok = ok && tc::mbar_wait_sleep(&sm.empty[i % NRING], (uint32_t)((i / NRING - 1) & 1));
        if (!ok) break;  // a wait gave up: request nothing more (the CTA ends soon)
        issue(i);
      }
    }
  } else if (warp == NCW) {
    // ================================================================ MMA issuer
    // Order of issue (= order of execution on the tensor core): the chain
    // K dh' -> (Y formed) -> w^T Y -> (dh formed) runs as soon as its operands
    // are written; Q^T (gamma dO) fills the gap while Y is formed and the next
    // chunk's P^T dO the gap while dh is formed.  After each product its tile
    // slot is released to the producer by a commit to the slot's empty barrier.
    if (lane == 0) {
      auto wait_tile = [&](int i) { ok = ok && tc::mbar_wait_sleep(&sm.full[i % NRING], (i / NRING) & 1); };
      auto slot_of = [&](int i) { return smem_u32(sm.slot[i % NRING]); };
      auto release = [&](int i) { tc::commit(&sm.empty[i % NRING]); };
      auto issue_p = [&](int ci) {  // P^T dO of chunk ci (its dO images are written)
        wait_tile(ci * TPC);  // (tile first)
        ok = ok && tc::mbar_wait_sleep(&sm.barO, (uint32_t)(ci & 1));
        tc::fence_after();
        tc::gemm_amn_k128(tmem + C_P, slot_of(ci * TPC), smem_u32(sm.Ot), SW, false);
        release(ci * TPC);  // (the commit after the chunk's K dh' covers it)
      };
      if (withO && !SPLIT) issue_p(0);
      for (int ci = 0; ci < n; ++ci) {
        const uint32_t par = (uint32_t)(ci & 1);
        const int t0 = ci * TPC;
        const int iQ = t0 + 1, iK = t0 + (withO ? 2 : 0), iW = t0 + (withO ? 3 : 1);
        // (each tile is waited for before the compute threads' signal, which comes later)
        wait_tile(iK);
        ok = ok && tc::mbar_wait_sleep(&sm.barXt, par);  // dh' image of this chunk
        tc::fence_after();
        tc::gemm_k128(tmem + C_Y, slot_of(iK), smem_u32(sm.Xt), SW, false);
        tc::commit(&sm.barY);
        release(iK);
        if (withO && !SPLIT) {
          wait_tile(iQ);
          tc::fence_after();
          tc::gemm_amn_k128(tmem + c_q(ci), slot_of(iQ), smem_u32(sm.Ogt), SW, false);
          tc::commit(&sm.barQ);
          release(iQ);
        }
        // (SPLIT: Q^T (gamma dO), issued by the other warp, has completed)
        if (withO && SPLIT) ok = ok && tc::mbar_wait_sleep(&sm.barQ, par);
        wait_tile(iW);
        ok = ok && tc::mbar_wait_sleep(&sm.barYt, par);  // (-Y)^T written
        tc::fence_after();
        tc::gemm_amn_k128(tmem + c_q(ci), slot_of(iW), smem_u32(sm.Yt), SW, withO);
        tc::commit(&sm.barH);
        release(iW);
        if (withO && !SPLIT && ci + 1 < n) issue_p(ci + 1);
      }
    }
  } else {
    // ========================================================== compute threads
    finish_gates(part, 0);
    if (withO) {
      if (DOTMA) {  // chunk index 0's rows (plain loads) into its slice buffer, for P^T dO
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(dO_slice(0) + tc::sw64_chunk(r, q)) = don[q];
      }
      write_do_images(don);
      tc::fence_proxy_async();
      tc::fence_before();
      arrive(&sm.barO);
    }
    arrive(&sm.barXt);  // the first dh' image was written before the block barrier
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32u * g32;  // lanes of this warp, its columns
    for (int ci = 0; ci < n; ++ci) {
      const int c = chunk_of(ci);
      const uint32_t par = (uint32_t)(ci & 1);
      // staging set ci % NSTAGE (dh', dDelta) was last read by the stores of chunk ci - NSTAGE
      const int set = ci % NSTAGE, use = ci / NSTAGE;
      uint4 dn[4];  // dO rows of chunk ci + 1: their images are written in this iteration
      if (!DOTMA) load_do(ci + 1, dn);
      if (!FOLD && use >= 1) ok = ok && tc::mbar_wait_sleep(&sm.sempty[set], (uint32_t)((use - 1) & 1));
      if (!FOLD && a.dstates) stage_row<SW>(sm.stage[set][0], r, g32, x);
      part = scan_part(gate_of(gnext, ci + 1), ci + 1);  // gates of the next chunk
      gnext = load_g(ci + 2);

      // ---- Y = diag(ef) K dh' + P^T dO (both complete on barY) ------------------------
      float y[32];
      ok = ok && tc::mbar_wait_sleep(&sm.barY, par);
      tc::fence_after();
      tc::ld32(tl + C_Y, y);
#pragma unroll
      for (int q = 0; q < 32; ++q) y[q] *= ef_r;
      if (withO) {  // (P^T dO has completed too: barY)
        float pd[32];
        tc::ld32(tl + C_P, pd);
#pragma unroll
        for (int q = 0; q < 32; ++q) y[q] += pd[q];
      }
#pragma unroll
      for (int q = 0; q < 32; ++q) y[q] = -y[q];
      write_bt_column<SW>(sm.Yt, r, 32 * g32, y);  // the chain's operand first
      tc::fence_proxy_async();
      tc::fence_before();
      arrive(&sm.barYt);
      if (!FOLD && a.ddelta) {
#pragma unroll
        for (int q = 0; q < 32; ++q) y[q] = -y[q];
        stage_row<SW>(sm.stage[set][1], r, g32, y);
      }
      if (!FOLD) {  // dh' and dDelta of this chunk are staged
        tc::fence_proxy_async();
        arrive(&sm.sfull[set]);
      }

      // ---- gates and dO images of the next chunk -------------------------------------
      const float gC_cur = gC;
      asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
      finish_gates(part, ci + 1);
      if (withO && ci + 1 < n) {  // both dO products of this chunk have read the images
        ok = ok && tc::mbar_wait_sleep(&sm.barQ, par);
        if (DOTMA) {  // the slice of chunk index ci + 1 (load number ci of dOt)
          ok = ok && tc::mbar_wait_sleep(&sm.barDO, par);
#pragma unroll
          for (int q = 0; q < 4; ++q) dn[q] = *reinterpret_cast<const uint4*>(dO_slice(ci + 1) + tc::sw64_chunk(r, q));
        }
        write_do_images(dn);
        tc::fence_proxy_async();
        tc::fence_before();
        arrive(&sm.barO);
      }

      // ---- dh = gamma_C dh' + Q^T (gamma dO) - w^T Y ---------------------------------
      ok = ok && tc::mbar_wait_sleep(&sm.barH, par);
      tc::fence_after();
      float hv[32];
      tc::ld32(tl + c_q(ci), hv);
#pragma unroll
      for (int q = 0; q < 32; ++q) x[q] = gC_cur * x[q] + hv[q];
      if (ci + 1 < n) {
        write_bt_column<SW>(sm.Xt, r, 32 * g32, x);
        tc::fence_proxy_async();
        tc::fence_before();
        arrive(&sm.barXt);
      }
    }
    if (FOLD) {
      store_row_f32((partA ? a.pairA : a.pairB) + ((bh * a.S + seg) * HD + r) * HD + col0, x);
    } else if (a.dh0 && seg == 0) {
      store_row_f32(a.dh0 + (bh * HD + r) * HD + col0, x);
    }
  }
  if (!ok && a.status) atomicOr(a.status, 1);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, Cfg::TMEM_COLS);
}

}  // namespace walkb
}  // namespace gdn
