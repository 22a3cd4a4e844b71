// kernels_a4d_f16_trace.cu -- f16 instantiations of the a4d chain kernels
// (kernel_units.cuh) with the event trace compiled in.
#define B2B_TRACE 1
#include "kernel_units.cuh"

namespace b2b {
namespace B2B_KNS {
template const void* variant_func_a4d<false>(Variant v);
template cudaError_t launch_variant_a4d<false>(Variant v, const CUtensorMap& a,
                                               const CUtensorMap& w0, const CUtensorMap& w1,
                                               const CUtensorMap& out, const ChainParams& p,
                                               int grid, size_t smem, cudaStream_t s);
}  // namespace B2B_KNS
}  // namespace b2b
