// kernels_cta2.cu -- fp16 and bf16 instantiations of the CTA-pair chain kernel
// (kernels_cta2_units.cuh), without the event trace.
#include "kernels_cta2_units.cuh"

namespace b2b {
namespace B2B_KNS {
template const void* cta2_func<false>();
template const void* cta2_func<true>();
template cudaError_t cta2_launch<false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                        const CUtensorMap&, const ChainParams&, int, size_t,
                                        cudaStream_t);
template cudaError_t cta2_launch<true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                       const CUtensorMap&, const ChainParams&, int, size_t,
                                       cudaStream_t);
template cudaError_t cta2_clusters<false>(size_t, int*);
template cudaError_t cta2_clusters<true>(size_t, int*);
template const void* pool2_func<false>();
template const void* pool2_func<true>();
template cudaError_t pool2_launch<false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                         const CUtensorMap&, const ChainParams&, int, size_t,
                                         cudaStream_t);
template cudaError_t pool2_launch<true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                        const CUtensorMap&, const ChainParams&, int, size_t,
                                        cudaStream_t);
template cudaError_t pool2_clusters<false>(size_t, int*);
template cudaError_t pool2_clusters<true>(size_t, int*);
}  // namespace B2B_KNS
}  // namespace b2b
