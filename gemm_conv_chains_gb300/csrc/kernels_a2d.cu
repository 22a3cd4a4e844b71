// kernels_a2d.cu -- instantiations of the chain kernel with a 2-D (row-major) A operand.
#include "chain_kernel.cuh"
#include "launch.h"

namespace b2b {

template <int MODE, bool A4D, bool W0MN, bool W1MN>
static cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                              const CUtensorMap& out, const ChainParams& p, int grid, size_t smem,
                              cudaStream_t stream) {
  chain_kernel<MODE, A4D, W0MN, W1MN><<<grid, kNumThreads, smem, stream>>>(a, w0, w1, out, p);
  return cudaGetLastError();
}

const void* variant_func_a2d(Variant v) {
  switch (v) {
    case V_GEMM_CHAIN: return reinterpret_cast<const void*>(&chain_kernel<MODE_CHAIN, false, true, true>);
    case V_CONV1X1_CHAIN: return reinterpret_cast<const void*>(&chain_kernel<MODE_CHAIN, false, false, false>);
    case V_GEMM_SINGLE: return reinterpret_cast<const void*>(&chain_kernel<MODE_SINGLE, false, true, false>);
    case V_CONV1X1_SINGLE: return reinterpret_cast<const void*>(&chain_kernel<MODE_SINGLE, false, false, false>);
    default: return nullptr;
  }
}

cudaError_t launch_variant_a2d(Variant v, const CUtensorMap& a, const CUtensorMap& w0,
                               const CUtensorMap& w1, const CUtensorMap& out, const ChainParams& p,
                               int grid, size_t smem, cudaStream_t s) {
  switch (v) {
    case V_GEMM_CHAIN: return launch_one<MODE_CHAIN, false, true, true>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV1X1_CHAIN: return launch_one<MODE_CHAIN, false, false, false>(a, w0, w1, out, p, grid, smem, s);
    case V_GEMM_SINGLE: return launch_one<MODE_SINGLE, false, true, false>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV1X1_SINGLE: return launch_one<MODE_SINGLE, false, false, false>(a, w0, w1, out, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace b2b
