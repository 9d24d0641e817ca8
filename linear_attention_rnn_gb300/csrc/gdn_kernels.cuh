// gdn_kernels.cuh -- argument blocks and launchers of the gated-delta-rule kernels
// (internal to the library; the public boundary is include/gdn.h).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "gdn_common.cuh"

namespace gdn {

// Per-chunk UT/WY preparation: persistent CTAs over (batch row, chunk, key head, value head) units.
struct PrepArgs {
  const bf16* q;
  const bf16* k;
  const bf16* v;
  const float* g;
  const float* beta;
  bf16* W;       // [BH][NC][CH][HD]  w = T diag(beta gamma) K      (nullable)
  bf16* U;       // [BH][NC][CH][HD]  u = T diag(beta) V            (nullable)
  bf16* P;       // [BH][NC][CH][CH]  (Q K^T) * decay, incl. diag   (nullable)
  bf16* Tb;      // [BH][NC][CH][CH]  T in bf16 (backward)           (nullable)
  float* S_dbg;  // [BH][NC][CH][CH]  fp32 S  (debug export)        (nullable)
  float* T_dbg;  // [BH][NC][CH][CH]  fp32 T  (debug export)        (nullable)
  int* status;   // bit 0 set if a bounded wait gave up (nullable)
  float* nrm;    // non-null: q, k are raw rows; prep normalises its K and Q tiles in shared
                 // memory and writes 1/||k||, 1/||q|| per row here, [B][Hk][NC][2][CH]
  int gate_logits;         // 1: g and beta hold logits a, b (g = -softplus(a), beta = sigmoid(b))
  int c64;                 // 1: 64-token chunks, two to a 128-row tile (block-diagonal S, T and P;
                           //    the gates restart at row 64)
  int B, T, Hk, Hv, NC;    // NC: 128-row tiles per sequence
};

// Sequential forward walk over the chunks of one segment for one
// (state-column slice, segment, batch*value head).
struct WalkFwdArgs {
  const bf16* W;
  const bf16* U;
  const bf16* P;
  const bf16* q;
  const bf16* k;
  const float* g;
  const float* hstart;     // entering state of each segment, fp32 (nullable = 0)
  long hstart_seg_stride;  // elements between consecutive segments' states
  long hstart_bh_stride;   // elements between consecutive (b, j)
  bf16* o;                 // [B,T,Hv,HD] (nullable)
  float* hT;               // [BH][HD][HD] written by the last segment (nullable)
  bf16* states;            // [BH][NC][HD][HD] bf16 entering state of every chunk (nullable)
  bf16* delta;             // [BH][NC][CH][HD] bf16 Delta of every chunk (nullable)
  float* pairA;            // fold output [BH][S][HD][HD]
  float* pairB;            // fold output [BH][S][HD][HD]
  int* status;             // bit 0 set if a bounded wait gave up (nullable)
  const float* nrm;        // non-null: K and Q tiles are raw rows, these their 1/||.|| (as PrepArgs)
  int gate_logits;         // 1: g and beta hold logits a, b (g = -softplus(a), beta = sigmoid(b))
  int c64;                 // 1: 64-token chunks (w, u, P, nrm in the preparation's 128-row tiles)
  int B, T, Hk, Hv, NC, S;  // NC: chunks per sequence (of 128 or 64 tokens)
  int NT;                  // 128-row tiles per sequence in w, u, P and nrm
};

// State columns per CTA of the forward walk's recompute mode (the output walk
// and the segment fold keep 32): a 64-column slice halves the CTAs for about
// 20% more time per chunk.
constexpr int WALK_STATES_SW = 64;

// TMA tensor maps of the forward walk: K and Q over [B, T, Hk, 128] (boxes of
// 64 columns x 128 tokens, 128-byte swizzle; 64 tokens with 64-token chunks),
// w and P over the workspace rows (same boxes); stores of WALK_STATES_SW-column
// slices of the entering states and Delta over the workspace rows.
struct WalkFwdMaps {
  CUtensorMap k, q, W, P;
  CUtensorMap St, De;
};

// Sequential backward walk (state cotangent) over the chunks of one segment.
struct WalkBwdArgs {
  const bf16* W;
  const bf16* P;
  const bf16* q;
  const bf16* k;
  const bf16* dO;
  const float* g;
  const float* hstart;     // cotangent of the state leaving each segment (nullable = 0)
  long hstart_seg_stride;
  long hstart_bh_stride;
  float* dh0;              // [BH][HD][HD] written by segment 0 (nullable)
  bf16* dstates;           // [BH][NC][HD][HD] bf16 cotangent of the state leaving every chunk
  bf16* ddelta;            // [BH][NC][CH][HD] bf16 dDelta of every chunk
  float* pairA;            // fold output
  float* pairB;
  int* status;             // bit 0 set if a bounded wait gave up (nullable)
  int gate_logits;         // 1: g and beta hold logits a, b (g = -softplus(a), beta = sigmoid(b))
  int B, T, Hk, Hv, NC, S;
};

// State columns per CTA of the backward walk (the segment fold keeps 32): a
// 64-column slice halves the CTAs for about 20% more time per chunk.
constexpr int WALK_BWD_SW = 64;

// Tensor maps of the backward walk's tiles: k and q as for the forward walk,
// w and P over the workspace rows (64 columns x 128 rows, 128-byte swizzle).
struct WalkBwdMaps {
  CUtensorMap k, q, W, P;
  CUtensorMap Ds, Dd;  // stores: leaving-state cotangents and dDelta (WALK_BWD_SW-column slices)
  CUtensorMap dO;      // loads: 32-column slices of dO over 128 tokens (64-byte swizzle)
};

// Sequential affine walk X <- A_i X (+ B_i) over i (segment prefix / compose).
struct AffineWalkArgs {
  const float* A;      // [batch][n][HD][HD]
  const float* Bv;     // [batch][n][HD][dv] (nullable = 0)
  const float* init;   // [batch][HD][dv] initial B-part columns (nullable = 0)
  float* outA;         // inclusive mode: [batch][n][HD][HD]
  float* outB;         // [batch][n][HD][dv]
  int batch, n, dv;
  int with_A;          // 1: state is [A | B] starting from [I | 0] (compose)
  int exclusive;       // 1: write the state entering map i (else after it)
  int reverse;         // 1: walk i = n-1 .. 0
};

// Chunk-parallel gradients, one CTA per (chunk, value head, batch row).
struct GradArgs {
  const bf16* q;
  const bf16* k;
  const bf16* v;
  const float* g;
  const float* beta;
  const bf16* dO;
  const bf16* Tb;       // [BH][NC][CH][CH]
  const bf16* states;   // [BH][NC][HD][HD]  h entering chunk
  const bf16* dstates;  // [BH][NC][HD][HD]  cotangent of h leaving chunk
  const bf16* delta;    // [BH][NC][CH][HD]
  const bf16* ddelta;   // [BH][NC][CH][HD]
  bf16* dq;             // [B,T,Hk,HD]
  bf16* dk;             // [B,T,Hk,HD]
  bf16* dv;             // [B,T,Hv,HD]
  float* dg;            // [B,T,Hv]
  float* dbeta;         // [B,T,Hv]
  int* status;          // bit 0 set if a bounded wait gave up (nullable)
  int gate_logits;         // 1: g and beta hold logits a, b (g = -softplus(a), beta = sigmoid(b))
  int B, T, Hk, Hv, NC;
};

// Launches kernel k with programmatic stream serialization: its CTAs may start
// (and run up to their pdl_wait) while the previous kernel in the stream ends.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

size_t prep_smem_bytes();
size_t grad_smem_bytes();

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
// The forward walk: its segment fold (fold = 1) or the walk with output.
cudaError_t launch_walk_fwd(const WalkFwdArgs& a, const WalkFwdMaps& m, int fold, cudaStream_t s);
// The backward walk on 32-column slices: its segment fold (fold = 1), or the
// walk alone (fold = 0; the maps' dh' and dDelta stores have 32-column boxes).
cudaError_t launch_walk_bwd(const WalkBwdArgs& a, const WalkBwdMaps& m, int fold, cudaStream_t s);
// The forward walk's recompute mode and the backward walk (fold = 0 both) in one launch.
cudaError_t launch_walk_pair(const WalkFwdArgs& fa, const WalkFwdMaps& fm, const WalkBwdArgs& ba,
                             const WalkBwdMaps& bm, cudaStream_t s);
cudaError_t launch_affine_walk(const AffineWalkArgs& a, cudaStream_t s);
// Element-wise layer operations on rows of HD bf16 values (gdn_layer.cu).
cudaError_t launch_l2norm(const bf16* x, bf16* y, long rows, float eps, cudaStream_t s);
cudaError_t launch_l2norm_bwd(const bf16* x, const bf16* dy, bf16* dx, long rows, float eps, cudaStream_t s);
cudaError_t launch_out_gate(const bf16* o, const bf16* z, bf16* y, long rows, cudaStream_t s);
cudaError_t launch_out_gate_bwd(const bf16* o, const bf16* z, const bf16* dy, bf16* dO, bf16* dz, long rows,
                                cudaStream_t s);
// (A, B) = (I, 0) for n [HD x HD] fp32 pairs (A nullable).
cudaError_t launch_identity_pairs(float* A, float* Bv, long n, cudaStream_t s);
cudaError_t launch_grads(const GradArgs& a, cudaStream_t s);
cudaError_t launch_selftest_wait(long long limit_ns, int* status, cudaStream_t s);

}  // namespace gdn
