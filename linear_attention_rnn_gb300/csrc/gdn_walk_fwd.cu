// gdn_walk_fwd.cu -- kernels of the sequential forward walk (the body is in
// gdn_walk_fwd.cuh): the segment fold and the walk with output, for 128- and
// 64-token chunks.  The state
// recompute of the backward runs in gdn_walk_pair.cu, beside the backward walk.
#include "gdn_walk_fwd.cuh"

namespace gdn {

namespace {

// (the walk with output and staged exports runs one more warp, the stores')
template <bool FOLD, bool STAGED, int SW, bool C64>
__global__ void __launch_bounds__(walkf::FwdCfg<SW>::NT + 32, 1)
    k_walk_fwd(WalkFwdArgs a, const __grid_constant__ WalkFwdMaps mp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  walkf::walk<FOLD, STAGED, SW, C64>(a, mp, base, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <bool FOLD, bool STAGED, int SW, bool C64 = false>
cudaError_t launch_one(const WalkFwdArgs& a, const WalkFwdMaps& m, cudaStream_t s) {
  const size_t smem = sizeof(walkf::WalkSmem<SW>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_walk_fwd<FOLD, STAGED, SW, C64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int NSL = HD / SW;
  const int nt = walkf::FwdCfg<SW>::NT + ((STAGED && a.o) ? 32 : 0);
  return launch_pdl(k_walk_fwd<FOLD, STAGED, SW, C64>, dim3(FOLD ? 2 * NSL : NSL, a.S, a.B * a.Hv), dim3(nt), smem,
                    s, a, m);
}

}  // namespace

cudaError_t launch_walk_fwd(const WalkFwdArgs& a, const WalkFwdMaps& m, int fold, cudaStream_t s) {
  if (a.c64) {  // 64-token chunks: the fold, or the walk with output (no exports)
    if (fold) return launch_one<true, false, 32, true>(a, m, s);
    if (!a.o || a.states || a.delta) return cudaErrorInvalidValue;
    return launch_one<false, false, 32, true>(a, m, s);
  }
  if (fold) return launch_one<true, false, 32>(a, m, s);
  // with output; with the entering states and Delta also (for a backward that
  // reads them), staged and stored by TMA as the recompute mode does (which
  // runs in the pair launch)
  if (!a.o) return cudaErrorInvalidValue;
  if (a.states || a.delta) return launch_one<false, true, 32>(a, m, s);
  return launch_one<false, false, 32>(a, m, s);
}

}  // namespace gdn
