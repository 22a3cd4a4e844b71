// kernels_a4d.cu -- instantiations of the chain kernel with the implicit-GEMM conv A operand.
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

const void* variant_func_a4d(Variant v) {
  switch (v) {
    case V_CONV_CHAIN: return reinterpret_cast<const void*>(&chain_kernel<MODE_CHAIN, true, false, false>);
    case V_CONV_SINGLE: return reinterpret_cast<const void*>(&chain_kernel<MODE_SINGLE, true, false, false>);
    case V_CONV_POOL: return reinterpret_cast<const void*>(&chain_kernel<MODE_POOL, true, false, false>);
    default: return nullptr;
  }
}

cudaError_t launch_variant_a4d(Variant v, const CUtensorMap& a, const CUtensorMap& w0,
                               const CUtensorMap& w1, const CUtensorMap& out, const ChainParams& p,
                               int grid, size_t smem, cudaStream_t s) {
  switch (v) {
    case V_CONV_CHAIN: return launch_one<MODE_CHAIN, true, false, false>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV_SINGLE: return launch_one<MODE_SINGLE, true, false, false>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV_POOL: return launch_one<MODE_POOL, true, false, false>(a, w0, w1, out, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace b2b
