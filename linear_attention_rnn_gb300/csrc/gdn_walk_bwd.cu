// gdn_walk_bwd.cu -- the segment fold of the reverse walk of the state
// cotangent (the body is in gdn_walk_bwd.cuh; gdn_walk_pair.cu runs the walk
// itself beside the forward state recompute).
#include "gdn_walk_bwd.cuh"

namespace gdn {

namespace {

// (one warp more than the walk's configuration: the dO products' issuer)
template <bool FOLD, int SW>
__global__ void __launch_bounds__(walkb::BwdCfg<SW>::NT + 32, 1)
    k_walk_bwd(WalkBwdArgs a, const __grid_constant__ WalkBwdMaps mp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  walkb::walk<FOLD, SW, true>(a, mp, base, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <bool FOLD, int SW>
cudaError_t launch_one(const WalkBwdArgs& a, const WalkBwdMaps& m, cudaStream_t s) {
  const size_t smem = sizeof(walkb::WalkBwdSmem<SW>) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(k_walk_bwd<FOLD, SW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int NSL = HD / SW;
  return launch_pdl(k_walk_bwd<FOLD, SW>, dim3(FOLD ? 2 * NSL : NSL, a.S, a.B * a.Hv),
                    dim3(walkb::BwdCfg<SW>::NT + 32), smem, s, a, m);
}

}  // namespace

cudaError_t launch_walk_bwd(const WalkBwdArgs& a, const WalkBwdMaps& m, int fold, cudaStream_t s) {
  // both on 32-column slices: the fold, or the walk alone (when the states it
  // needs beside it were kept by the forward; otherwise it runs in the pair launch)
  if (fold) return launch_one<true, 32>(a, m, s);
  return launch_one<false, 32>(a, m, s);
}

}  // namespace gdn
