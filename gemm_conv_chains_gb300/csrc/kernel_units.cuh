// kernel_units.cuh -- the compiled instantiations of the chain kernel, per operand dtype.
// Each kernels_<a2d|a4d>_<dtype>.cu instantiates one group, so the units compile in
// parallel and every kernel holds the epilogue of one dtype only.
#pragma once

#include "chain_kernel.cuh"
#include "launch.h"

namespace b2b {
namespace B2B_KNS {

template <int MODE, bool A4D, bool W0MN, bool W1MN, bool BF16, bool WIDE = false,
          bool PAIR = false, bool NOPAIR = false, bool W0RES = false, bool TWO = false>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(
      &chain_kernel<MODE, A4D, W0MN, W1MN, BF16, WIDE, PAIR, NOPAIR, W0RES, TWO>);
}

template <int MODE, bool A4D, bool W0MN, bool W1MN, bool BF16, bool WIDE = false,
          bool PAIR = false, bool NOPAIR = false, bool W0RES = false, bool TWO = false>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                       const CUtensorMap& out, const ChainParams& p, int grid, size_t smem,
                       cudaStream_t stream) {
  return launch_chain(chain_kernel<MODE, A4D, W0MN, W1MN, BF16, WIDE, PAIR, NOPAIR, W0RES, TWO>, a, w0,
                      w1, out, p, grid, smem, stream, chain_threads(MODE, TWO));
}

// 2-D A operand: GEMM chains (row-major weights) and 1x1 convs (K-major filters).
template <bool BF16>
const void* variant_func_a2d(Variant v) {
  switch (v) {
    case V_GEMM_CHAIN: return kernel_ptr<MODE_CHAIN, false, true, true, BF16>();
    case V_CONV1X1_CHAIN: return kernel_ptr<MODE_CHAIN, false, false, false, BF16>();
    case V_GEMM_SINGLE: return kernel_ptr<MODE_SINGLE, false, true, false, BF16>();
    case V_CONV1X1_SINGLE: return kernel_ptr<MODE_SINGLE, false, false, false, BF16>();
    case V_GEMM_CHAIN3: return kernel_ptr<MODE_CHAIN3, false, true, true, BF16>();
    case V_GEMM_CHAIN_WIDE: return kernel_ptr<MODE_CHAIN, false, true, true, BF16, true>();
    case V_GEMM_CHAIN_PAIR: return kernel_ptr<MODE_CHAIN, false, true, true, BF16, false, true>();
    case V_GEMM_CHAIN_PAIR_W0:
      return kernel_ptr<MODE_CHAIN, false, true, true, BF16, false, true, false, true>();
    case V_GEMM_CHAIN_NP:
      return kernel_ptr<MODE_CHAIN, false, true, true, BF16, false, false, true>();
    case V_CONV1X1_CHAIN_NP:
      return kernel_ptr<MODE_CHAIN, false, false, false, BF16, false, false, true>();
    default: return nullptr;
  }
}

template <bool BF16>
cudaError_t launch_variant_a2d(Variant v, const CUtensorMap& a, const CUtensorMap& w0,
                               const CUtensorMap& w1, const CUtensorMap& out,
                               const ChainParams& p, int grid, size_t smem, cudaStream_t s) {
  switch (v) {
    case V_GEMM_CHAIN:
      return launch_one<MODE_CHAIN, false, true, true, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV1X1_CHAIN:
      return launch_one<MODE_CHAIN, false, false, false, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_GEMM_SINGLE:
      return launch_one<MODE_SINGLE, false, true, false, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV1X1_SINGLE:
      return launch_one<MODE_SINGLE, false, false, false, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_GEMM_CHAIN3:
      return launch_one<MODE_CHAIN3, false, true, true, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_GEMM_CHAIN_WIDE:
      return launch_one<MODE_CHAIN, false, true, true, BF16, true>(a, w0, w1, out, p, grid, smem,
                                                                   s);
    case V_GEMM_CHAIN_PAIR:
      return launch_one<MODE_CHAIN, false, true, true, BF16, false, true>(a, w0, w1, out, p, grid,
                                                                         smem, s);
    case V_GEMM_CHAIN_PAIR_W0:
      return launch_one<MODE_CHAIN, false, true, true, BF16, false, true, false, true>(
          a, w0, w1, out, p, grid, smem, s);
    case V_GEMM_CHAIN_NP:
      return launch_one<MODE_CHAIN, false, true, true, BF16, false, false, true>(
          a, w0, w1, out, p, grid, smem, s);
    case V_CONV1X1_CHAIN_NP:
      return launch_one<MODE_CHAIN, false, false, false, BF16, false, false, true>(
          a, w0, w1, out, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

// 4-D A operand: implicit-GEMM convs (chain, single, conv + max-pool).
template <bool BF16>
const void* variant_func_a4d(Variant v) {
  switch (v) {
    case V_CONV_CHAIN: return kernel_ptr<MODE_CHAIN, true, false, false, BF16>();
    case V_CONV_CHAIN_NP:
      return kernel_ptr<MODE_CHAIN, true, false, false, BF16, false, false, true>();
    case V_CONV_SINGLE: return kernel_ptr<MODE_SINGLE, true, false, false, BF16>();
    case V_CONV_POOL: return kernel_ptr<MODE_POOL, true, false, false, BF16>();
    case V_CONV_CHAIN_2I:
      return kernel_ptr<MODE_CHAIN, true, false, false, BF16, false, false, false, false, true>();
    default: return nullptr;
  }
}

template <bool BF16>
cudaError_t launch_variant_a4d(Variant v, const CUtensorMap& a, const CUtensorMap& w0,
                               const CUtensorMap& w1, const CUtensorMap& out,
                               const ChainParams& p, int grid, size_t smem, cudaStream_t s) {
  switch (v) {
    case V_CONV_CHAIN:
      return launch_one<MODE_CHAIN, true, false, false, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV_CHAIN_NP:
      return launch_one<MODE_CHAIN, true, false, false, BF16, false, false, true>(
          a, w0, w1, out, p, grid, smem, s);
    case V_CONV_SINGLE:
      return launch_one<MODE_SINGLE, true, false, false, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV_POOL:
      return launch_one<MODE_POOL, true, false, false, BF16>(a, w0, w1, out, p, grid, smem, s);
    case V_CONV_CHAIN_2I:
      return launch_one<MODE_CHAIN, true, false, false, BF16, false, false, false, false, true>(
          a, w0, w1, out, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace B2B_KNS
}  // namespace b2b
