// gdn_walk_pair.cu -- the backward's two sequential walks in one launch.
//
// The state recompute (the forward walk in its recompute mode) and the reverse
// walk of the state cotangent need nothing from each other: both read only the
// preparation's tiles, the inputs and their own entering values.  Each is a
// chain of dependent per-chunk products that keeps its SMs far from their
// peak, so the two run side by side on different SMs of one launch, each on
// 64-column state slices (half the CTAs of a 32-column walk): 2 + 2 CTAs per
// (segment, batch row, value head).
#include "gdn_walk_bwd.cuh"
#include "gdn_walk_fwd.cuh"

namespace gdn {

namespace {

constexpr int PAIR_NT = walkf::FwdCfg<WALK_STATES_SW>::NT;
static_assert(PAIR_NT == walkb::BwdCfg<WALK_BWD_SW>::NT, "both walks run with one block size");
constexpr int NF = HD / WALK_STATES_SW, NB = HD / WALK_BWD_SW;  // state slices of each walk
constexpr size_t PAIR_SMEM = (sizeof(walkf::WalkSmem<WALK_STATES_SW>) > sizeof(walkb::WalkBwdSmem<WALK_BWD_SW>)
                                  ? sizeof(walkf::WalkSmem<WALK_STATES_SW>)
                                  : sizeof(walkb::WalkBwdSmem<WALK_BWD_SW>)) +
                             1024;

// CTAs x < NB walk the cotangent (the longer walk, scheduled first); the others
// recompute the entering states and Delta.
__global__ void __launch_bounds__(PAIR_NT, 1)
    k_walk_pair(WalkFwdArgs fa, const __grid_constant__ WalkFwdMaps fm, WalkBwdArgs ba,
                const __grid_constant__ WalkBwdMaps bm) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  if ((int)blockIdx.x < NB)
    walkb::walk<false, WALK_BWD_SW>(ba, bm, base, blockIdx.x, blockIdx.y, blockIdx.z);
  else
    walkf::walk<false, true, WALK_STATES_SW>(fa, fm, base, blockIdx.x - NB, blockIdx.y, blockIdx.z);
}

}  // namespace

cudaError_t launch_walk_pair(const WalkFwdArgs& fa, const WalkFwdMaps& fm, const WalkBwdArgs& ba,
                             const WalkBwdMaps& bm, cudaStream_t s) {
  if (fa.S != ba.S || fa.B != ba.B || fa.Hv != ba.Hv || fa.NC != ba.NC || fa.o) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_walk_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PAIR_SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_walk_pair, dim3(NB + NF, fa.S, fa.B * fa.Hv), dim3(PAIR_NT), PAIR_SMEM, s, fa, fm, ba, bm);
}

}  // namespace gdn
