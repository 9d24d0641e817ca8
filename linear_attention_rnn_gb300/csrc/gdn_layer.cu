// gdn_layer.cu -- the element-wise operations around the chunked rule in a
// GatedDeltaNet layer: per-token L2 normalisation of q and k before the rule,
// and the output gate y = o * silu(z) after it, with their backward passes.
// (The gate activations beta = sigmoid(b) and g = -softplus(a) are applied by
// the rule's own kernels where they load the gates; see gate_act.)
//
// The pages name these operations only through the layer's buffers: the
// "qkvz" activations [B, T, H, D] of PR "Shard the GatedDeltaNet sequence
// under ici_context_parallelism" (description), of which q and k enter the
// rule normalised and z gates its output.
//
// Every kernel streams rows of 128 bf16 values: one warp per row, four values
// (8 bytes) per lane, fp32 arithmetic, grid-stride over the rows.
#include "gdn_kernels.cuh"

namespace gdn {

namespace {

constexpr int RW = 8;  // rows (warps) per 256-thread block

__device__ __forceinline__ void load4(const bf16* p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y);
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
}
__device__ __forceinline__ void store4(bf16* p, const float (&x)[4]) {
  uint2 u;
  u.x = pack_bf16(x[0], x[1]);
  u.y = pack_bf16(x[2], x[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// y = x / sqrt(sum x^2 + eps) per row
__global__ void __launch_bounds__(32 * RW) k_l2norm(const bf16* x, bf16* y, long rows, float eps) {
  const int lane = threadIdx.x & 31;
  for (long r = (long)blockIdx.x * RW + (threadIdx.x >> 5); r < rows; r += (long)gridDim.x * RW) {
    float v[4];
    load4(x + r * HD + 4 * lane, v);
    const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
    const float inv = rsqrtf(ss + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] *= inv;
    store4(y + r * HD + 4 * lane, v);
  }
}

// dx = (dy - y (y . dy)) / sqrt(sum x^2 + eps), y = x / sqrt(sum x^2 + eps)
__global__ void __launch_bounds__(32 * RW) k_l2norm_bwd(const bf16* x, const bf16* dy, bf16* dx, long rows,
                                                        float eps) {
  const int lane = threadIdx.x & 31;
  for (long r = (long)blockIdx.x * RW + (threadIdx.x >> 5); r < rows; r += (long)gridDim.x * RW) {
    float v[4], d[4];
    load4(x + r * HD + 4 * lane, v);
    load4(dy + r * HD + 4 * lane, d);
    const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
    const float inv = rsqrtf(ss + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] *= inv;  // y
    const float yd = warp_sum(v[0] * d[0] + v[1] * d[1] + v[2] * d[2] + v[3] * d[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = inv * (d[i] - v[i] * yd);
    store4(dx + r * HD + 4 * lane, d);
  }
}

__device__ __forceinline__ float sigm(float z) { return 1.f / (1.f + expf(-z)); }

// y = o * silu(z), silu(z) = z sigmoid(z)
__global__ void __launch_bounds__(32 * RW) k_out_gate(const bf16* o, const bf16* z, bf16* y, long rows) {
  const int lane = threadIdx.x & 31;
  for (long r = (long)blockIdx.x * RW + (threadIdx.x >> 5); r < rows; r += (long)gridDim.x * RW) {
    float ov[4], zv[4];
    load4(o + r * HD + 4 * lane, ov);
    load4(z + r * HD + 4 * lane, zv);
#pragma unroll
    for (int i = 0; i < 4; ++i) ov[i] *= zv[i] * sigm(zv[i]);
    store4(y + r * HD + 4 * lane, ov);
  }
}

// dO = dy * silu(z),  dz = dy * o * silu'(z),  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
__global__ void __launch_bounds__(32 * RW) k_out_gate_bwd(const bf16* o, const bf16* z, const bf16* dy, bf16* dO,
                                                          bf16* dz, long rows) {
  const int lane = threadIdx.x & 31;
  for (long r = (long)blockIdx.x * RW + (threadIdx.x >> 5); r < rows; r += (long)gridDim.x * RW) {
    float ov[4], zv[4], dv[4], a[4], b[4];
    load4(o + r * HD + 4 * lane, ov);
    load4(z + r * HD + 4 * lane, zv);
    load4(dy + r * HD + 4 * lane, dv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float s = sigm(zv[i]);
      a[i] = dv[i] * zv[i] * s;
      b[i] = dv[i] * ov[i] * s * (1.f + zv[i] * (1.f - s));
    }
    store4(dO + r * HD + 4 * lane, a);
    store4(dz + r * HD + 4 * lane, b);
  }
}

int row_blocks(long rows) {
  const long b = (rows + RW - 1) / RW;
  return (int)(b < 152 * 16 ? (b > 0 ? b : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_l2norm(const bf16* x, bf16* y, long rows, float eps, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_l2norm<<<row_blocks(rows), 32 * RW, 0, s>>>(x, y, rows, eps);
  return cudaGetLastError();
}

cudaError_t launch_l2norm_bwd(const bf16* x, const bf16* dy, bf16* dx, long rows, float eps, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_l2norm_bwd<<<row_blocks(rows), 32 * RW, 0, s>>>(x, dy, dx, rows, eps);
  return cudaGetLastError();
}

cudaError_t launch_out_gate(const bf16* o, const bf16* z, bf16* y, long rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_out_gate<<<row_blocks(rows), 32 * RW, 0, s>>>(o, z, y, rows);
  return cudaGetLastError();
}

cudaError_t launch_out_gate_bwd(const bf16* o, const bf16* z, const bf16* dy, bf16* dO, bf16* dz, long rows,
                                cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_out_gate_bwd<<<row_blocks(rows), 32 * RW, 0, s>>>(o, z, dy, dO, dz, rows);
  return cudaGetLastError();
}

}  // namespace gdn
