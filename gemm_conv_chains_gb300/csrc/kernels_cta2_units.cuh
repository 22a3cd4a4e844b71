// kernels_cta2_units.cuh -- the compiled instantiations of the CTA-pair chain kernel, per
// operand dtype (see kernels_cta2.cu / kernels_cta2_trace.cu).
#pragma once

#include "chain_cta2_kernel.cuh"
#include "chain_cta2_pool_kernel.cuh"
#include "launch.h"

namespace b2b {
namespace B2B_KNS {

template <bool BF16>
const void* cta2_func() {
  return reinterpret_cast<const void*>(&chain_cta2_kernel<BF16>);
}

template <bool BF16>
cudaError_t cta2_launch(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                        const CUtensorMap& out, const ChainParams& p, int grid, size_t smem,
                        cudaStream_t s) {
  return launch_chain_cta2(chain_cta2_kernel<BF16>, a, w0, w1, out, p, grid, smem, s);
}

template <bool BF16>
cudaError_t cta2_clusters(size_t smem, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(static_cast<unsigned>(kNumThreads));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, chain_cta2_kernel<BF16>, &cfg);
}

// The conv + pool kernel over CTA pairs: the same launch shape.
template <bool BF16>
const void* pool2_func() {
  return reinterpret_cast<const void*>(&chain_cta2_pool_kernel<BF16>);
}

template <bool BF16>
cudaError_t pool2_launch(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                         const CUtensorMap& out, const ChainParams& p, int grid, size_t smem,
                         cudaStream_t s) {
  return launch_chain_cta2(chain_cta2_pool_kernel<BF16>, a, w0, w1, out, p, grid, smem, s,
                           kPool2Threads);
}

template <bool BF16>
cudaError_t pool2_clusters(size_t smem, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(static_cast<unsigned>(kPool2Threads));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, chain_cta2_pool_kernel<BF16>, &cfg);
}

}  // namespace B2B_KNS
}  // namespace b2b
