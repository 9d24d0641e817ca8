// gdn_api.cu -- the extern "C" boundary declared in include/gdn.h: argument
// validation (on the host, before anything is enqueued), workspace layout,
// and the launch sequence of each operation on the caller's stream.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "gdn.h"
#include "gdn_kernels.cuh"
#include "gdn_tmap.cuh"

using namespace gdn;

namespace {

constexpr size_t ALIGN = 256;
inline size_t up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// C: tokens per chunk (128, or 64 in the forward); NC chunks per sequence; the
// per-chunk tiles (w, u, P, ...) are stored in NT 128-row tiles per sequence,
// two 64-token chunks to a tile.
struct Dims {
  int B, T, Hk, Hv, NC, S, C, NT;
  long BH() const { return (long)B * Hv; }
};

// chunk = 64 only where the caller allows it (the forward entry points)
int check_dims(int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int n_segments, bool allow64 = false) {
  if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || n_segments < 0) return GDN_ERR_ARG;
  if (Hv % Hk != 0) return GDN_ERR_ARG;
  if (dk != HD || dv != HD || !(chunk == CH || (allow64 && chunk == 64))) return GDN_ERR_SHAPE;
  return GDN_OK;
}

Dims make_dims(int B, int T, int Hk, int Hv, int n_segments, int chunk = CH) {
  Dims d;
  d.B = B;
  d.T = T;
  d.Hk = Hk;
  d.Hv = Hv;
  d.C = chunk;
  d.NC = (T + chunk - 1) / chunk;
  d.NT = (T + CH - 1) / CH;
  int S = n_segments == 0 ? gdn_default_segments(B, T, Hv, chunk) : n_segments;
  if (S > d.NC) S = d.NC;
  if (S < 1) S = 1;
  d.S = S;
  return d;
}

// Workspace layout.  Forward: w, u, P per chunk; with segments also the
// per-segment (A, B) pairs and entering states.  Backward adds T (bf16), the
// bf16 entering states, Delta, the state cotangents, dDelta and the fp32
// per-value-head dq/dk.
struct Layout {
  size_t status, W, U, P, Tb, pairA, pairB, hin, dhin, states, delta, dstates, ddelta, total;
};

Layout layout(const Dims& d, bool bwd) {
  Layout L;
  memset(&L, 0, sizeof L);
  const size_t chunks = (size_t)d.BH() * d.NT;  // 128-row tiles
  const size_t tile = (size_t)CH * HD * sizeof(bf16);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += up(bytes);
    return o;
  };
  L.status = take(sizeof(int));  // bit 0 set by a kernel whose bounded wait gave up
  L.W = take(chunks * tile);
  L.U = take(chunks * tile);
  L.P = take(chunks * tile);
  if (d.S > 1) {
    const size_t pair = (size_t)d.BH() * d.S * HD * HD * sizeof(float);
    L.pairA = take(pair);
    L.pairB = take(pair);
    L.hin = take(pair);
  }
  if (bwd) {
    if (d.S > 1) L.dhin = take((size_t)d.BH() * d.S * HD * HD * sizeof(float));  // entering cotangents
    L.Tb = take(chunks * tile);
    L.states = take(chunks * tile);
    L.delta = take(chunks * tile);
    L.dstates = take(chunks * tile);
    L.ddelta = take(chunks * tile);
  }
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// The per-chunk quantities of the UT/WY preparation (w, u, P and, for the
// backward, T): in the workspace, or in a caller's buffer that a forward fills
// and the backward of the same inputs reads instead of recomputing them.
struct Tiles {
  bf16 *W, *U, *P, *Tb;
  bf16 *states, *delta;  // the state entering every chunk and Delta (backward)
  float* hin;            // with segments: the state entering every segment, [B Hv][S][128][128] fp32
};

Tiles ws_tiles(void* ws, const Layout& L) {
  Tiles t;
  t.W = at<bf16>(ws, L.W);
  t.U = at<bf16>(ws, L.U);
  t.P = at<bf16>(ws, L.P);
  t.Tb = L.Tb ? at<bf16>(ws, L.Tb) : nullptr;
  t.states = L.states ? at<bf16>(ws, L.states) : nullptr;
  t.delta = L.delta ? at<bf16>(ws, L.delta) : nullptr;
  t.hin = L.hin ? at<float>(ws, L.hin) : nullptr;
  return t;
}

// saved buffer: w, u, P, T, the entering state of every chunk and Delta, each
// [B Hv][NC][128][128] bf16, and with segments the entering state of every
// segment, [B Hv][S][128][128] fp32
size_t saved_total(const Dims& d) {
  const size_t part = up((size_t)d.BH() * d.NC * CH * HD * sizeof(bf16));
  return 6 * part + (d.S > 1 ? up((size_t)d.BH() * d.S * HD * HD * sizeof(float)) : 0);
}

Tiles saved_tiles(void* saved, const Dims& d) {
  const size_t part = up((size_t)d.BH() * d.NC * CH * HD * sizeof(bf16));
  Tiles t;
  t.W = at<bf16>(saved, 0);
  t.U = at<bf16>(saved, part);
  t.P = at<bf16>(saved, 2 * part);
  t.Tb = at<bf16>(saved, 3 * part);
  t.states = at<bf16>(saved, 4 * part);
  t.delta = at<bf16>(saved, 5 * part);
  t.hin = d.S > 1 ? at<float>(saved, 6 * part) : nullptr;
  return t;
}

// swizzle of a stored [128 x sw] bf16 walk slice: its rows are 2 sw bytes
CUtensorMapSwizzle slice_swizzle(int sw) { return sw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// Records the caller's events after each launch (timing variants only).
struct Marks {
  void* const* ev;
  int n;
  int i;
  cudaStream_t s;
  int rec() {
    if (ev && i < n && ev[i]) {
      cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
      ++i;
      return cuda_status(e);
    }
    ++i;
    return GDN_OK;
  }
};

// Forward walk set-up: prep has run.  Fills the walk's arguments and tensor
// maps; with segments it also runs the fold and the cross-segment prefix, so
// that the walk (launched by the caller) replays every segment from its
// entering state.
// hin_ready: the segments' entering states are already in tl.hin (a forward
// kept them), so the fold and the prefix are not run again.
// The exports (states, delta) are stored in slices of 32 columns by the walk
// with output, of WALK_STATES_SW columns by the recompute beside the reverse walk.
int prepare_forward_walk(const Dims& d, const Layout& Lw, void* ws, const Tiles& tl, const void* q,
                         const void* k, const float* g, const float* h0, void* o, float* hT,
                         bf16* states, bf16* delta, int gate_logits, bool hin_ready, cudaStream_t s,
                         Marks& mk, WalkFwdArgs& w, WalkFwdMaps& mp, const float* nrm = nullptr) {
  const int esw = o ? 32 : WALK_STATES_SW;
  memset(&w, 0, sizeof w);
  w.gate_logits = gate_logits;
  w.nrm = nrm;
  w.W = tl.W;
  w.U = tl.U;
  w.P = tl.P;
  w.q = static_cast<const bf16*>(q);
  w.k = static_cast<const bf16*>(k);
  w.g = g;
  w.B = d.B;
  w.T = d.T;
  w.Hk = d.Hk;
  w.Hv = d.Hv;
  w.NC = d.NC;
  w.NT = d.NT;
  w.c64 = d.C == 64;
  w.S = d.S;
  w.o = static_cast<bf16*>(o);
  w.hT = hT;
  w.states = states;
  w.delta = delta;
  w.status = at<int>(ws, Lw.status);
  memset(&mp, 0, sizeof mp);
  const uint64_t wrows = (uint64_t)d.BH() * d.NT * CH;
  const uint32_t box = (uint32_t)d.C;  // tokens (rows) per TMA box: one chunk
  if (!tmap_heads(&mp.k, k, d.B, d.T, d.Hk, HD, box) || !tmap_heads(&mp.q, q, d.B, d.T, d.Hk, HD, box) ||
      !tmap_2d(&mp.W, w.W, HD, wrows, HD * sizeof(bf16), 64, box, true) ||
      !tmap_2d(&mp.P, w.P, CH, wrows, CH * sizeof(bf16), 64, box, true) ||
      (states && !tmap_2d_sw(&mp.St, states, HD, wrows, HD * sizeof(bf16), esw, CH, slice_swizzle(esw))) ||
      (delta && !tmap_2d_sw(&mp.De, delta, HD, wrows, HD * sizeof(bf16), esw, CH, slice_swizzle(esw))))
    return GDN_ERR_CUDA;
  if (d.S == 1) {
    w.hstart = h0;
    w.hstart_bh_stride = (long)HD * HD;
    w.hstart_seg_stride = 0;
    return GDN_OK;
  }
  if (hin_ready) {
    w.hstart = tl.hin;
    w.hstart_bh_stride = (long)d.S * HD * HD;
    w.hstart_seg_stride = (long)HD * HD;
    return GDN_OK;
  }
  WalkFwdArgs f = w;
  f.pairA = at<float>(ws, Lw.pairA);
  f.pairB = at<float>(ws, Lw.pairB);
  f.o = nullptr;
  f.hT = nullptr;
  f.states = nullptr;
  f.delta = nullptr;
  int rc = cuda_status(launch_walk_fwd(f, mp, 1, s));
  if (rc || (rc = mk.rec())) return rc;
  AffineWalkArgs x;
  memset(&x, 0, sizeof x);
  x.A = f.pairA;
  x.Bv = f.pairB;
  x.init = h0;
  x.outB = tl.hin;
  x.batch = (int)d.BH();
  x.n = d.S;
  x.dv = HD;
  x.with_A = 0;
  x.exclusive = 1;
  x.reverse = 0;
  rc = cuda_status(launch_affine_walk(x, s));
  if (rc || (rc = mk.rec())) return rc;
  w.hstart = tl.hin;
  w.hstart_bh_stride = (long)d.S * HD * HD;
  w.hstart_seg_stride = (long)HD * HD;
  return GDN_OK;
}

}  // namespace

extern "C" {

const char* gdn_strerror(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_ARG: return "invalid argument (null pointer, misalignment, negative size or Hv % Hk != 0)";
    case GDN_ERR_SHAPE:
      return "unsupported shape (d_k = d_v = 128; chunk = 128, or 64 in the forward entry points)";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    case GDN_ERR_CUDA: return "CUDA launch failed";
    case GDN_ERR_TIMEOUT: return "a bounded in-kernel wait gave up";
    case GDN_ERR_UNSUPPORTED: return "unsupported device";
    default: return "unknown status";
  }
}

int gdn_default_segments(int B, int T, int Hv, int chunk) {
  if (chunk <= 0 || T <= 0 || B <= 0 || Hv <= 0) return 1;
  const long NC = (T + chunk - 1) / chunk;
  if (NC <= 64) return 1;
  // The one-segment walk runs 4 CTAs per (batch row, value head).  When those
  // keep a quarter of the SMs or more busy, segments only add work: the fold
  // pushes every chunk through the 256 columns of [A | B], and the prefix is
  // sequential over the segments.  Otherwise take enough segments for the fold
  // (8 CTAs per segment and head) to fill the SMs about twice, with at least
  // 8 chunks per segment.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 152;
  const long heads = (long)B * Hv;
  if (4 * heads * 4 >= sms) return 1;
  long S = (2L * sms + 8 * heads - 1) / (8 * heads);
  if (S > NC / 8) S = NC / 8;
  if (S > 256) S = 256;
  return S < 2 ? 2 : (int)S;
}

size_t gdn_fwd_workspace_bytes(int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk,
                               int n_segments) {
  if (check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments, true) != GDN_OK) return 0;
  return layout(make_dims(B, T, Hk, Hv, n_segments, chunk), false).total;
}

size_t gdn_bwd_workspace_bytes(int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk,
                               int n_segments) {
  if (check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments) != GDN_OK) return 0;
  return layout(make_dims(B, T, Hk, Hv, n_segments), true).total;
}

static int fwd_impl(const void* q, const void* k, const void* v, const float* g,
                    const float* beta, const float* h0, void* o, float* hT, int B, int T, int Hk,
                    int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                    size_t ws_bytes, void* stream, void* const* events, int n_events,
                    int gate_logits = 0, void* saved = nullptr, size_t saved_bytes = 0,
                    float* nrm = nullptr) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments, true);
  if (rc) return rc;
  if (saved && chunk != CH) return GDN_ERR_SHAPE;  // the backward takes 128-token chunks
  const long tokens = (long)B * T;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, h0, o, hT, ws, saved};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims d = make_dims(B, T, Hk, Hv, n_segments, chunk);
  if (B == 0) return GDN_OK;
  if (T == 0) {  // no tokens: the final state is the initial state
    if (!hT) return GDN_OK;
    const size_t bytes = (size_t)B * Hv * HD * HD * sizeof(float);
    return cuda_status(h0 ? cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, s)
                          : cudaMemsetAsync(hT, 0, bytes, s));
  }
  const Layout L = layout(d, false);
  if (!ws || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if (saved && saved_bytes < saved_total(d)) return GDN_ERR_WORKSPACE;
  Marks mk = {events, n_events, 0, s};
  if ((rc = cuda_status(cudaMemsetAsync(at<int>(ws, L.status), 0, sizeof(int), s)))) return rc;
  // with a saved buffer, prep's w, u and P go there, and T beside them, for the backward
  const Tiles tl = saved ? saved_tiles(saved, d) : ws_tiles(ws, L);

  PrepArgs p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const bf16*>(q);
  p.k = static_cast<const bf16*>(k);
  p.v = static_cast<const bf16*>(v);
  p.g = g;
  p.beta = beta;
  p.W = tl.W;
  p.U = tl.U;
  p.P = tl.P;
  p.Tb = saved ? tl.Tb : nullptr;
  p.nrm = nrm;  // raw q and k: prep scales its tiles' rows to unit length
  p.status = at<int>(ws, L.status);
  p.gate_logits = gate_logits;
  p.c64 = d.C == 64;
  p.B = B;
  p.T = T;
  p.Hk = Hk;
  p.Hv = Hv;
  p.NC = d.NT;
  rc = cuda_status(launch_prep(p, s));
  if (rc || (rc = mk.rec())) return rc;
  WalkFwdArgs w;
  WalkFwdMaps mp;
  // with a saved buffer the walk also keeps the entering state of every chunk and Delta
  if ((rc = prepare_forward_walk(d, L, ws, tl, q, k, g, h0, o, hT, saved ? tl.states : nullptr,
                                 saved ? tl.delta : nullptr, gate_logits, false, s, mk, w, mp, nrm)))
    return rc;
  if ((rc = cuda_status(launch_walk_fwd(w, mp, 0, s)))) return rc;
  return mk.rec();
}

static int bwd_impl(const void* q, const void* k, const void* v, const float* g,
                    const float* beta, const float* h0, const void* dO, const float* dhT,
                    void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0, int B,
                    int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                    size_t ws_bytes, void* stream, void* const* events, int n_events,
                    int gate_logits = 0, const void* saved = nullptr, size_t saved_bytes = 0) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments);
  if (rc) return rc;
  const long tokens = (long)B * T;
  if (tokens > 0 && (!q || !k || !v || !g || !beta || !dO || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, h0, dO, dhT, dq, dk, dv, dg, dbeta, dh0, ws, saved};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims d = make_dims(B, T, Hk, Hv, n_segments);
  if (B == 0) return GDN_OK;
  if (T == 0) {  // dh0 = dhT
    if (!dh0) return GDN_OK;
    const size_t bytes = (size_t)B * Hv * HD * HD * sizeof(float);
    return cuda_status(dhT ? cudaMemcpyAsync(dh0, dhT, bytes, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(dh0, 0, bytes, s));
  }
  const Layout L = layout(d, true);
  if (!ws || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if (saved && saved_bytes < saved_total(d)) return GDN_ERR_WORKSPACE;
  Marks mk = {events, n_events, 0, s};
  if ((rc = cuda_status(cudaMemsetAsync(at<int>(ws, L.status), 0, sizeof(int), s)))) return rc;
  const Tiles tl = saved ? saved_tiles(const_cast<void*>(saved), d) : ws_tiles(ws, L);

  // 1. per-chunk UT quantities (w, u, P, T), unless the forward kept them
  if (!saved) {
    PrepArgs p;
    memset(&p, 0, sizeof p);
    p.q = static_cast<const bf16*>(q);
    p.k = static_cast<const bf16*>(k);
    p.v = static_cast<const bf16*>(v);
    p.g = g;
    p.beta = beta;
    p.W = tl.W;
    p.U = tl.U;
    p.P = tl.P;
    p.Tb = tl.Tb;
    p.status = at<int>(ws, L.status);
    p.gate_logits = gate_logits;
    p.B = B;
    p.T = T;
    p.Hk = Hk;
    p.Hv = Hv;
    p.NC = d.NC;
    rc = cuda_status(launch_prep(p, s));
    if (rc || (rc = mk.rec())) return rc;
  }
  // 2. recompute of the state entering every chunk, and Delta (with segments:
  //    its fold and cross-segment prefix now, the replay below), unless the
  //    forward kept them
  WalkFwdArgs fw;
  WalkFwdMaps fm;
  if (!saved) {
    rc = prepare_forward_walk(d, L, ws, tl, q, k, g, h0, nullptr, nullptr, tl.states, tl.delta,
                              gate_logits, false, s, mk, fw, fm);
    if (rc) return rc;
  }
  // the reverse walk runs alone on 32-column slices when the forward kept the
  // states, else beside the recompute on WALK_BWD_SW-column slices
  const int bsw = saved ? 32 : WALK_BWD_SW;
  // 3. reverse walk of the state cotangent (with segments: its fold and prefix
  //    now); it needs nothing from the recompute, so the two walks run side by
  //    side in one launch
  WalkBwdArgs w;
  memset(&w, 0, sizeof w);
  w.W = tl.W;
  w.P = tl.P;
  w.q = static_cast<const bf16*>(q);
  w.k = static_cast<const bf16*>(k);
  w.dO = static_cast<const bf16*>(dO);
  w.g = g;
  w.B = B;
  w.T = T;
  w.Hk = Hk;
  w.Hv = Hv;
  w.NC = d.NC;
  w.S = d.S;
  w.dh0 = dh0;
  w.dstates = at<bf16>(ws, L.dstates);
  w.ddelta = at<bf16>(ws, L.ddelta);
  w.status = at<int>(ws, L.status);
  w.gate_logits = gate_logits;
  WalkBwdMaps bm;
  memset(&bm, 0, sizeof bm);
  {
    const uint64_t wrows = (uint64_t)d.BH() * d.NC * CH;
    if (!tmap_heads(&bm.k, k, d.B, d.T, d.Hk, HD) || !tmap_heads(&bm.q, q, d.B, d.T, d.Hk, HD) ||
        !tmap_2d(&bm.W, w.W, HD, wrows, HD * sizeof(bf16), 64, CH, true) ||
        !tmap_2d(&bm.P, w.P, CH, wrows, CH * sizeof(bf16), 64, CH, true) ||
        !tmap_2d_sw(&bm.Ds, w.dstates, HD, wrows, HD * sizeof(bf16), bsw, CH, slice_swizzle(bsw)) ||
        !tmap_2d_sw(&bm.Dd, w.ddelta, HD, wrows, HD * sizeof(bf16), bsw, CH, slice_swizzle(bsw)) ||
        !tmap_heads_box(&bm.dO, dO, d.B, d.T, d.Hv, HD, 32, CH, CU_TENSOR_MAP_SWIZZLE_64B))
      return GDN_ERR_CUDA;
  }
  if (d.S == 1) {
    w.hstart = dhT;
    w.hstart_bh_stride = (long)HD * HD;
    w.hstart_seg_stride = 0;
  } else {
    WalkBwdArgs f = w;
    f.pairA = at<float>(ws, L.pairA);
    f.pairB = at<float>(ws, L.pairB);
    f.dh0 = nullptr;
    rc = cuda_status(launch_walk_bwd(f, bm, 1, s));
    if (rc || (rc = mk.rec())) return rc;
    AffineWalkArgs x;
    memset(&x, 0, sizeof x);
    x.A = f.pairA;
    x.Bv = f.pairB;
    x.init = dhT;
    x.outB = at<float>(ws, L.dhin);
    x.batch = (int)d.BH();
    x.n = d.S;
    x.dv = HD;
    x.with_A = 0;
    x.exclusive = 1;
    x.reverse = 1;
    rc = cuda_status(launch_affine_walk(x, s));
    if (rc || (rc = mk.rec())) return rc;
    w.hstart = at<float>(ws, L.dhin);
    w.hstart_bh_stride = (long)d.S * HD * HD;
    w.hstart_seg_stride = (long)HD * HD;
  }
  if (saved)
    rc = cuda_status(launch_walk_bwd(w, bm, 0, s));
  else
    rc = cuda_status(launch_walk_pair(fw, fm, w, bm, s));
  if (rc || (rc = mk.rec())) return rc;
  // 4. chunk-parallel gradients (dq and dk summed over the value heads of each key head)
  GradArgs ga;
  memset(&ga, 0, sizeof ga);
  ga.q = static_cast<const bf16*>(q);
  ga.k = static_cast<const bf16*>(k);
  ga.v = static_cast<const bf16*>(v);
  ga.g = g;
  ga.beta = beta;
  ga.dO = static_cast<const bf16*>(dO);
  ga.Tb = tl.Tb;
  ga.states = tl.states;
  ga.dstates = at<bf16>(ws, L.dstates);
  ga.delta = tl.delta;
  ga.ddelta = at<bf16>(ws, L.ddelta);
  ga.dq = static_cast<bf16*>(dq);
  ga.dk = static_cast<bf16*>(dk);
  ga.status = at<int>(ws, L.status);
  ga.gate_logits = gate_logits;
  ga.dv = static_cast<bf16*>(dv);
  ga.dg = dg;
  ga.dbeta = dbeta;
  ga.B = B;
  ga.T = T;
  ga.Hk = Hk;
  ga.Hv = Hv;
  ga.NC = d.NC;
  rc = cuda_status(launch_grads(ga, s));
  return rc ? rc : mk.rec();
}

size_t gdn_saved_bytes(int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments) {
  if (check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments) != GDN_OK) return 0;
  return saved_total(make_dims(B, T, Hk, Hv, n_segments));
}

int gdn_chunk_fwd_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     const float* h0, void* o, float* hT, int B, int T, int Hk, int Hv, int d_k,
                     int d_v, int chunk, int n_segments, void* saved, size_t saved_bytes, void* ws,
                     size_t ws_bytes, void* stream, void* const* events, int n_events) {
  return fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, Hk, Hv, d_k, d_v, chunk, n_segments, ws,
                  ws_bytes, stream, events, n_events, 0, saved, saved_bytes);
}

int gdn_chunk_bwd_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     const float* h0, const void* dO, const float* dhT, void* dq, void* dk, void* dv,
                     float* dg, float* dbeta, float* dh0, int B, int T, int Hk, int Hv, int d_k,
                     int d_v, int chunk, int n_segments, const void* saved, size_t saved_bytes,
                     void* ws, size_t ws_bytes, void* stream, void* const* events, int n_events) {
  return bwd_impl(q, k, v, g, beta, h0, dO, dhT, dq, dk, dv, dg, dbeta, dh0, B, T, Hk, Hv, d_k,
                  d_v, chunk, n_segments, ws, ws_bytes, stream, events, n_events, 0, saved,
                  saved_bytes);
}

int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const float* h0, void* o, float* hT, int B, int T, int Hk, int Hv, int d_k,
                  int d_v, int chunk, int n_segments, void* ws, size_t ws_bytes, void* stream) {
  return fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, Hk, Hv, d_k, d_v, chunk, n_segments, ws,
                  ws_bytes, stream, nullptr, 0);
}

int gdn_chunk_fwd_timed(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* h0, void* o, float* hT, int B, int T,
                        int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                        size_t ws_bytes, void* stream, void* const* events, int n_events) {
  return fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, Hk, Hv, d_k, d_v, chunk, n_segments, ws,
                  ws_bytes, stream, events, n_events);
}

int gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const float* h0, const void* dO, const float* dhT, void* dq, void* dk, void* dv,
                  float* dg, float* dbeta, float* dh0, int B, int T, int Hk, int Hv, int d_k,
                  int d_v, int chunk, int n_segments, void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(q, k, v, g, beta, h0, dO, dhT, dq, dk, dv, dg, dbeta, dh0, B, T, Hk, Hv, d_k,
                  d_v, chunk, n_segments, ws, ws_bytes, stream, nullptr, 0);
}

int gdn_chunk_bwd_timed(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* h0, const void* dO, const float* dhT,
                        void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0, int B,
                        int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments,
                        void* ws, size_t ws_bytes, void* stream, void* const* events,
                        int n_events) {
  return bwd_impl(q, k, v, g, beta, h0, dO, dhT, dq, dk, dv, dg, dbeta, dh0, B, T, Hk, Hv, d_k,
                  d_v, chunk, n_segments, ws, ws_bytes, stream, events, n_events);
}

// ---- layer entry points: normalised q/k, gate logits, output gate -------------------
// Workspace of a layer call: the rule's own workspace first (so that its
// status word is the first word, as gdn_workspace_status reads it), then the
// normalised q and k (bf16, [B, T, Hk, 128] each), a [B, T, Hv, 128] bf16
// buffer (forward: the rule's output when the caller keeps none; backward:
// the rule's output cotangent), and for the backward the cotangents of the
// normalised q and k.
struct LayerLayout {
  size_t core, nrm, qn, kn, obuf, dO, dqn, dkn, total;
};

static LayerLayout layer_layout(int backward, int B, int T, int Hk, int Hv, int n_segments, int chunk) {
  LayerLayout L;
  memset(&L, 0, sizeof L);
  const size_t qk = (size_t)B * T * Hk * HD * sizeof(bf16);
  const size_t vv = (size_t)B * T * Hv * HD * sizeof(bf16);
  const Dims d = make_dims(B, T, Hk, Hv, n_segments, chunk);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += up(bytes);
    return o;
  };
  L.core = take(layout(d, backward != 0).total);
  if (backward) {  // normalised copies of q and k, and their cotangents
    L.qn = take(qk);
    L.kn = take(qk);
    L.obuf = take(vv);
    L.dO = L.obuf;
    L.dqn = take(qk);
    L.dkn = take(qk);
  } else {  // the rows' 1/||k||, 1/||q|| (the forward normalises inside its kernels)
    L.nrm = take((size_t)B * Hk * d.NT * 2 * CH * sizeof(float));
    L.obuf = take(vv);
  }
  L.total = off;
  return L;
}

constexpr float kL2Eps = 1e-6f;

size_t gdn_layer_workspace_bytes(int backward, int B, int T, int Hk, int Hv, int d_k, int d_v,
                                 int chunk, int n_segments) {
  if (check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments, !backward) != GDN_OK) return 0;
  return layer_layout(backward, B, T, Hk, Hv, n_segments, chunk).total;
}

int gdn_layer_fwd(const void* q, const void* k, const void* v, const float* a, const float* b,
                  const void* z, const float* h0, void* y, void* o, float* hT, int B, int T, int Hk,
                  int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws, size_t ws_bytes,
                  void* stream) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments, true);
  if (rc) return rc;
  const long tokens = (long)B * T;
  if (tokens > 0 && (!q || !k || !v || !a || !b || !y)) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, a, b, z, h0, y, o, hT, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ARG;
  if (B == 0) return GDN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0)  // no tokens: the final state is the initial state
    return fwd_impl(q, k, v, a, b, h0, y, hT, B, T, Hk, Hv, d_k, d_v, chunk, n_segments, nullptr, 0,
                    stream, nullptr, 0, 1);
  const LayerLayout L = layer_layout(0, B, T, Hk, Hv, n_segments, chunk);
  if (!ws || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  // the rule's output: straight into y without a gate, else into o (or the workspace);
  // q and k go in raw: the preparation normalises the rows of its K and Q tiles and
  // the walk scales by the same 1/||k||, 1/||q|| where it reads them
  void* core_o = !z ? y : (o ? o : at<void>(ws, L.obuf));
  rc = fwd_impl(q, k, v, a, b, h0, core_o, hT, B, T, Hk, Hv, d_k, d_v, chunk, n_segments,
                at<void>(ws, L.core), L.nrm - L.core, stream, nullptr, 0, 1, nullptr, 0,
                at<float>(ws, L.nrm));
  if (rc) return rc;
  if (z) {
    rc = cuda_status(launch_out_gate(static_cast<const bf16*>(core_o), static_cast<const bf16*>(z),
                                     static_cast<bf16*>(y), tokens * Hv, s));
    if (rc) return rc;
  } else if (o) {
    rc = cuda_status(cudaMemcpyAsync(o, y, (size_t)tokens * Hv * HD * sizeof(bf16),
                                     cudaMemcpyDeviceToDevice, s));
  }
  return rc;
}

int gdn_layer_bwd(const void* q, const void* k, const void* v, const float* a, const float* b,
                  const void* z, const float* h0, const void* o, const void* dy, const float* dhT,
                  void* dq, void* dk, void* dv, float* da, float* db, void* dz, float* dh0, int B,
                  int T, int Hk, int Hv, int d_k, int d_v, int chunk, int n_segments, void* ws,
                  size_t ws_bytes, void* stream) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments);
  if (rc) return rc;
  const long tokens = (long)B * T;
  if (tokens > 0 && (!q || !k || !v || !a || !b || !dy || !dq || !dk || !dv || !da || !db))
    return GDN_ERR_ARG;
  if (tokens > 0 && z && (!o || !dz)) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, a, b, z, h0, o, dy, dhT, dq, dk, dv, da, db, dz, dh0, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ARG;
  if (B == 0) return GDN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0)
    return bwd_impl(q, k, v, a, b, h0, dy, dhT, dq, dk, dv, da, db, dh0, B, T, Hk, Hv, d_k, d_v, chunk,
                    n_segments, nullptr, 0, stream, nullptr, 0, 1);
  const LayerLayout L = layer_layout(1, B, T, Hk, Hv, n_segments, CH);
  if (!ws || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  bf16* qn = at<bf16>(ws, L.qn);
  bf16* kn = at<bf16>(ws, L.kn);
  bf16* dqn = at<bf16>(ws, L.dqn);
  bf16* dkn = at<bf16>(ws, L.dkn);
  if ((rc = cuda_status(launch_l2norm(static_cast<const bf16*>(q), qn, tokens * Hk, kL2Eps, s)))) return rc;
  if ((rc = cuda_status(launch_l2norm(static_cast<const bf16*>(k), kn, tokens * Hk, kL2Eps, s)))) return rc;
  const void* dO = dy;
  if (z) {  // the gate's backward gives the rule's output cotangent and dz
    bf16* dOb = at<bf16>(ws, L.dO);
    rc = cuda_status(launch_out_gate_bwd(static_cast<const bf16*>(o), static_cast<const bf16*>(z),
                                         static_cast<const bf16*>(dy), dOb, static_cast<bf16*>(dz),
                                         tokens * Hv, s));
    if (rc) return rc;
    dO = dOb;
  }
  rc = bwd_impl(qn, kn, v, a, b, h0, dO, dhT, dqn, dkn, dv, da, db, dh0, B, T, Hk, Hv, d_k, d_v, chunk,
                n_segments, at<void>(ws, L.core), L.qn - L.core, stream, nullptr, 0, 1);
  if (rc) return rc;
  if ((rc = cuda_status(launch_l2norm_bwd(static_cast<const bf16*>(q), dqn, static_cast<bf16*>(dq),
                                          tokens * Hk, kL2Eps, s))))
    return rc;
  return cuda_status(launch_l2norm_bwd(static_cast<const bf16*>(k), dkn, static_cast<bf16*>(dk), tokens * Hk,
                                       kL2Eps, s));
}

int gdn_affine_compose(const float* A, const float* B, float* A_out, float* B_out, int batch,
                       int n, int d_k, int d_v, void* stream) {
  if (batch < 0 || n < 0) return GDN_ERR_ARG;
  if (d_k != HD || d_v <= 0 || d_v > HD || d_v % 16 != 0) return GDN_ERR_SHAPE;
  if ((long)batch * n == 0) return GDN_OK;
  if (!A || !B || !A_out || !B_out) return GDN_ERR_ARG;
  const void* ptrs[] = {A, B, A_out, B_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return GDN_ERR_ARG;
  AffineWalkArgs x;
  memset(&x, 0, sizeof x);
  x.A = A;
  x.Bv = B;
  x.init = nullptr;
  x.outA = A_out;
  x.outB = B_out;
  x.batch = batch;
  x.n = n;
  x.dv = d_v;
  x.with_A = 1;
  x.exclusive = 0;
  x.reverse = 0;
  return cuda_status(launch_affine_walk(x, static_cast<cudaStream_t>(stream)));
}

int gdn_segment_fold(const void* k, const void* v, const float* g, const float* beta,
                     float* A_out, float* B_out, int B, int T, int Hk, int Hv, int d_k, int d_v,
                     int chunk, int n_segments, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, n_segments, true);
  if (rc) return rc;
  const int NC = (T + chunk - 1) / chunk;
  if (n_segments < 1 || n_segments > (NC > 1 ? NC : 1)) return GDN_ERR_ARG;
  if (B == 0) return GDN_OK;
  if (!B_out) return GDN_ERR_ARG;
  if (T > 0 && (!k || !v || !g || !beta)) return GDN_ERR_ARG;
  const void* ptrs[] = {k, v, g, beta, A_out, B_out, ws};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) return cuda_status(launch_identity_pairs(A_out, B_out, (long)B * Hv, s));
  const Dims d = make_dims(B, T, Hk, Hv, 1, chunk);
  const Layout L = layout(d, false);
  if (!ws || ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  if ((rc = cuda_status(cudaMemsetAsync(at<int>(ws, L.status), 0, sizeof(int), s)))) return rc;
  // w and u of every chunk (no output, so no P)
  PrepArgs p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const bf16*>(k);  // unused: P is not requested
  p.k = static_cast<const bf16*>(k);
  p.v = static_cast<const bf16*>(v);
  p.g = g;
  p.beta = beta;
  p.W = at<bf16>(ws, L.W);
  p.U = at<bf16>(ws, L.U);
  p.status = at<int>(ws, L.status);
  p.c64 = chunk == 64;
  p.B = B;
  p.T = T;
  p.Hk = Hk;
  p.Hv = Hv;
  p.NC = d.NT;
  if ((rc = cuda_status(launch_prep(p, s)))) return rc;
  // pass 1 of the segment scan: each segment's chunks pushed through [A | B] from [I | 0]
  WalkFwdArgs f;
  memset(&f, 0, sizeof f);
  f.W = p.W;
  f.U = p.U;
  f.P = at<bf16>(ws, L.P);
  f.q = static_cast<const bf16*>(k);
  f.k = static_cast<const bf16*>(k);
  f.g = g;
  f.B = B;
  f.T = T;
  f.Hk = Hk;
  f.Hv = Hv;
  f.NC = NC;
  f.NT = d.NT;
  f.c64 = chunk == 64;
  f.S = n_segments;
  f.pairA = A_out;
  f.pairB = B_out;
  f.status = p.status;
  WalkFwdMaps mp;
  memset(&mp, 0, sizeof mp);
  const uint64_t wrows = (uint64_t)d.BH() * d.NT * CH;
  const uint32_t box = (uint32_t)chunk;
  if (!tmap_heads(&mp.k, k, B, T, Hk, HD, box) || !tmap_heads(&mp.q, k, B, T, Hk, HD, box) ||
      !tmap_2d(&mp.W, f.W, HD, wrows, HD * sizeof(bf16), 64, box, true) ||
      !tmap_2d(&mp.P, f.P, CH, wrows, CH * sizeof(bf16), 64, box, true))
    return GDN_ERR_CUDA;
  return cuda_status(launch_walk_fwd(f, mp, 1, s));
}

int gdn_debug_ut(const void* k, const void* v, const float* g, const float* beta, float* S_out,
                 float* T_out, void* w_out, void* u_out, int B, int T, int Hk, int Hv, int d_k,
                 int d_v, int chunk, void* stream) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, 1, true);
  if (rc) return rc;
  if ((long)B * T == 0) return GDN_OK;
  if (!k || !v || !g || !beta) return GDN_ERR_ARG;
  const void* ptrs[] = {k, v, g, beta, S_out, T_out, w_out, u_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return GDN_ERR_ARG;
  PrepArgs p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const bf16*>(k);  // unused: P is not requested
  p.k = static_cast<const bf16*>(k);
  p.v = static_cast<const bf16*>(v);
  p.g = g;
  p.beta = beta;
  p.W = static_cast<bf16*>(w_out);
  p.U = static_cast<bf16*>(u_out);
  p.S_dbg = S_out;
  p.T_dbg = T_out;
  p.c64 = chunk == 64;
  p.B = B;
  p.T = T;
  p.Hk = Hk;
  p.Hv = Hv;
  p.NC = (T + CH - 1) / CH;  // 128-row tiles
  return cuda_status(launch_prep(p, static_cast<cudaStream_t>(stream)));
}

int gdn_workspace_status(const void* ws, void* stream) {
  if (!ws) return GDN_ERR_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
  int st = 0;  // the status word is the first field of every workspace layout
  if (cudaMemcpy(&st, ws, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  return (st & 1) ? GDN_ERR_TIMEOUT : GDN_OK;
}

int gdn_selftest_wait_timeout(long long limit_ns, int* status, void* stream) {
  if (!status || limit_ns < 1000LL || limit_ns > 10000000000LL) return GDN_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return GDN_ERR_CUDA;
  if (launch_selftest_wait(limit_ns, status, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  return (st & 1) ? GDN_ERR_TIMEOUT : GDN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward without any allocation.
//
// Some callers cannot hand this library a workspace and must not trigger an
// allocation: code that runs after a service has planned and locked all of
// its device memory (a cudaMalloc there could fail, fragment the plan, or
// stall every stream on the device while it synchronises), or hosts whose
// device memory belongs entirely to another framework that exposes no
// scratch buffer to plug-ins.  For them the forward below keeps its scratch
// (w, u and the masked Q K^T of every chunk) in one fixed array that lives in
// this library's device image.  Every GPU that loads the library holds the
// array until the process exits, which is why it is kept to a modest size.
namespace {

// one status word, then w, u and P of every unit (the forward workspace of
// gdn_chunk_fwd with one segment)
constexpr size_t kNoAllocScratchBytes =
    256 + (size_t)GDN_NOALLOC_MAX_UNITS * 3 * CH * HD * sizeof(bf16) + 3 * 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The name of a
// __device__ array in host code is only a host-side stand-in, so the address
// is looked up with the device current.  Outside stream capture it is looked
// up on every call (cheap once the module is loaded, and correct after the
// device's context was reset and the module reloaded at a new address);
// during a capture the address cached by the last call outside capture is used.
int noalloc_scratch(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  } else if (!g_noalloc_addr[dev]) {
    return GDN_ERR_CUDA;  // no call outside capture has looked the address up yet
  }
  *out = g_noalloc_addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" int gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                     const float* beta, const float* h0, void* o, float* hT,
                                     int B, int T, int Hk, int Hv, int d_k, int d_v, int chunk,
                                     void* stream) {
  int rc = check_dims(B, T, Hk, Hv, d_k, d_v, chunk, 1, true);
  if (rc) return rc;
  const long units = (long)B * Hv * ((T + CH - 1) / CH);  // 128-row tiles of w, u and P
  if (units > GDN_NOALLOC_MAX_UNITS) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (units > 0 && (rc = noalloc_scratch(static_cast<cudaStream_t>(stream), &scratch))) return rc;
  return fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, Hk, Hv, d_k, d_v, chunk, 1, scratch,
                  kNoAllocScratchBytes, stream, nullptr, 0);
}

// The status word of the fixed scratch array (its first 4 bytes, as in every
// workspace layout) after the last gdn_chunk_fwd_noalloc on the current device.
extern "C" int gdn_noalloc_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  int st = 0;
  if (cudaMemcpyFromSymbol(&st, g_noalloc_scratch, sizeof st, 0, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GDN_ERR_CUDA;
  return (st & 1) ? GDN_ERR_TIMEOUT : GDN_OK;
}
