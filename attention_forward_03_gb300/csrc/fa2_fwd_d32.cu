// Instantiations of the sm_103a forward kernel for head dimension 32 (in the layout of 64).
#include "fa2_kernel.cuh"

namespace fa2 {
template cudaError_t launch_fwd<32, false, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  const Params&, int, cudaStream_t);
template cudaError_t launch_fwd<32, false, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                 const Params&, int, cudaStream_t);
template cudaError_t launch_fwd<32, true, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                 const Params&, int, cudaStream_t);
template cudaError_t launch_fwd<32, true, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const Params&, int, cudaStream_t);
}  // namespace fa2
