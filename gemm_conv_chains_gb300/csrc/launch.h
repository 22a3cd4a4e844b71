// launch.h -- internal interface between the host API (api.cu) and the kernel units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernel_params.h"

namespace b2b {

// The compiled instantiations of the chain kernel.
//   GEMM_*     2-D A operand, weights W[K][N] row-major (MN-major B operand)
//   CONV1X1_*  2-D A operand (NHWC pixels as rows), weights W[Cout][Cin] (K-major)
//   CONV_*     4-D A operand (implicit GEMM per filter tap), weights W[Cout][R][S][Cin]
enum Variant : int {
  V_GEMM_CHAIN = 0,
  V_CONV1X1_CHAIN,
  V_CONV_CHAIN,
  V_GEMM_SINGLE,
  V_CONV1X1_SINGLE,
  V_CONV_SINGLE,
  V_CONV_POOL,
  V_GEMM_CHAIN3,
  V_GEMM_CHAIN_WIDE,
  V_GEMM_CHAIN_PAIR,   // P in TMEM, tiles in pairs, streamed weights (other loops left out)
  V_GEMM_CHAIN_NP,     // the chain variants above with P in shared memory (the P-in-TMEM
  V_CONV1X1_CHAIN_NP,  //   loops left out)
  V_CONV_CHAIN_NP,
  V_GEMM_CHAIN_PAIR_W0,   // tile pairs, P in TMEM, W0 resident, A and W1 streamed, output
                          //   stored from registers
  V_GEMM_CHAIN_CTA2,      // the chain over CTA pairs (chain_cta2_kernel.cuh)
  V_CONV_CHAIN_2I,        // conv chain, two MMA issuers, P in TMEM, output staged per warp
  V_CONV_POOL_CTA2,       // conv + pool over CTA pairs (chain_cta2_pool_kernel.cuh)
  V_COUNT
};

using ChainKernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, ChainParams);

// Launches a chain kernel with programmatic stream serialisation: the kernel may be
// scheduled while the previous kernel of the stream finishes, and it waits for that
// kernel (griddepcontrol.wait) before it touches global memory.
inline cudaError_t launch_chain(ChainKernelFn fn, const CUtensorMap& a, const CUtensorMap& w0,
                                const CUtensorMap& w1, const CUtensorMap& out,
                                const ChainParams& p, int grid, size_t smem,
                                cudaStream_t stream, int threads = kNumThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a, w0, w1, out, p);
}

// Launches a CTA-pair kernel (V_GEMM_CHAIN_CTA2) in clusters of two CTAs (`grid` even),
// with programmatic stream serialisation as launch_chain.
inline cudaError_t launch_chain_cta2(ChainKernelFn fn, const CUtensorMap& a, const CUtensorMap& w0,
                                     const CUtensorMap& w1, const CUtensorMap& out,
                                     const ChainParams& p, int grid, size_t smem,
                                     cudaStream_t stream, int threads = kNumThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, a, w0, w1, out, p);
}

// How many clusters of two CTAs of a CTA-pair kernel (the b2b GEMM chain's, or with `pool`
// the conv + pool one; dtype, build) can be resident at once with `smem` bytes of dynamic
// shared memory each (its function attributes set), or an error.
cudaError_t cta2_max_clusters(bool bf16, bool trace, size_t smem, int* clusters,
                              bool pool = false);

// Kernel function pointer of a variant, operand dtype and build (with or without the event
// trace), for cudaFuncSetAttribute.
const void* variant_func(Variant v, bool bf16, bool trace);

// Launches the variant's kernel for p.is_bf16, the traced build when p.trace is set.
cudaError_t launch_variant(Variant v, const CUtensorMap& a, const CUtensorMap& w0,
                           const CUtensorMap& w1, const CUtensorMap& out, const ChainParams& p,
                           int grid, size_t smem, cudaStream_t stream);

// Plain 2x2/2 max-pool over NHWC fp16/bf16 (the unfused pooling operator).
cudaError_t launch_maxpool(int is_bf16, int N, int H, int W, int C, const void* x, void* y,
                           int num_sms, cudaStream_t stream);

// Batch normalisation folded into weights [Co][K] (out_inner 0) or [K][Co] (out_inner 1)
// and bias [Co]; fp32 arithmetic, one rounding per stored value.
cudaError_t launch_fold_batchnorm(int is_bf16, int64_t Co, int64_t K, int out_inner,
                                  const void* Wt, const void* b, const float* gamma,
                                  const float* beta, const float* mean, const float* var,
                                  float eps, void* W_out, void* b_out, int num_sms,
                                  cudaStream_t stream);

// One-CTA kernel whose only wait can never complete; it must time out.
cudaError_t launch_probe_timeout(uint64_t limit_ns, uint32_t* err, cudaStream_t stream);

}  // namespace b2b
