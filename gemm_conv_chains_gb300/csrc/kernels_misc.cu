// kernels_misc.cu -- the plain max-pool operator of the unfused path, the timeout probe,
// and the variant dispatch over the two chain-kernel units.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace b2b {

// The kernel units, each compiled without (b2b::plain) and with (b2b::traced) the trace.
#define B2B_UNIT_DECLS                                                                       \
  template <bool BF16>                                                                       \
  const void* variant_func_a2d(Variant v);                                                   \
  template <bool BF16>                                                                       \
  const void* variant_func_a4d(Variant v);                                                   \
  template <bool BF16>                                                                       \
  cudaError_t launch_variant_a2d(Variant v, const CUtensorMap& a, const CUtensorMap& w0,     \
                                 const CUtensorMap& w1, const CUtensorMap& out,              \
                                 const ChainParams& p, int grid, size_t smem, cudaStream_t s); \
  template <bool BF16>                                                                       \
  cudaError_t launch_variant_a4d(Variant v, const CUtensorMap& a, const CUtensorMap& w0,     \
                                 const CUtensorMap& w1, const CUtensorMap& out,              \
                                 const ChainParams& p, int grid, size_t smem, cudaStream_t s); \
  template <bool BF16>                                                                       \
  const void* cta2_func();                                                                   \
  template <bool BF16>                                                                       \
  cudaError_t cta2_launch(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1, \
                          const CUtensorMap& out, const ChainParams& p, int grid, size_t smem, \
                          cudaStream_t s);                                                   \
  template <bool BF16>                                                                       \
  cudaError_t cta2_clusters(size_t smem, int* clusters);                                     \
  template <bool BF16>                                                                       \
  const void* pool2_func();                                                                  \
  template <bool BF16>                                                                       \
  cudaError_t pool2_launch(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1, \
                           const CUtensorMap& out, const ChainParams& p, int grid, size_t smem, \
                           cudaStream_t s);                                                  \
  template <bool BF16>                                                                       \
  cudaError_t pool2_clusters(size_t smem, int* clusters);
namespace plain {
B2B_UNIT_DECLS
}
namespace traced {
B2B_UNIT_DECLS
}
#undef B2B_UNIT_DECLS

static bool is_a4d(Variant v) {
  return v == V_CONV_CHAIN || v == V_CONV_CHAIN_NP || v == V_CONV_CHAIN_2I || v == V_CONV_SINGLE ||
         v == V_CONV_POOL;
}

const void* variant_func(Variant v, bool bf16, bool trace) {
  if (v == V_GEMM_CHAIN_CTA2) {
    if (trace) return bf16 ? traced::cta2_func<true>() : traced::cta2_func<false>();
    return bf16 ? plain::cta2_func<true>() : plain::cta2_func<false>();
  }
  if (v == V_CONV_POOL_CTA2) {
    if (trace) return bf16 ? traced::pool2_func<true>() : traced::pool2_func<false>();
    return bf16 ? plain::pool2_func<true>() : plain::pool2_func<false>();
  }
  if (trace) {
    if (is_a4d(v)) return bf16 ? traced::variant_func_a4d<true>(v) : traced::variant_func_a4d<false>(v);
    return bf16 ? traced::variant_func_a2d<true>(v) : traced::variant_func_a2d<false>(v);
  }
  if (is_a4d(v)) return bf16 ? plain::variant_func_a4d<true>(v) : plain::variant_func_a4d<false>(v);
  return bf16 ? plain::variant_func_a2d<true>(v) : plain::variant_func_a2d<false>(v);
}

cudaError_t launch_variant(Variant v, const CUtensorMap& a, const CUtensorMap& w0,
                           const CUtensorMap& w1, const CUtensorMap& out, const ChainParams& p,
                           int grid, size_t smem, cudaStream_t stream) {
  const bool bf16 = p.is_bf16 != 0;
  if (v == V_GEMM_CHAIN_CTA2) {
    if (p.trace != nullptr)
      return bf16 ? traced::cta2_launch<true>(a, w0, w1, out, p, grid, smem, stream)
                  : traced::cta2_launch<false>(a, w0, w1, out, p, grid, smem, stream);
    return bf16 ? plain::cta2_launch<true>(a, w0, w1, out, p, grid, smem, stream)
                : plain::cta2_launch<false>(a, w0, w1, out, p, grid, smem, stream);
  }
  if (v == V_CONV_POOL_CTA2) {
    if (p.trace != nullptr)
      return bf16 ? traced::pool2_launch<true>(a, w0, w1, out, p, grid, smem, stream)
                  : traced::pool2_launch<false>(a, w0, w1, out, p, grid, smem, stream);
    return bf16 ? plain::pool2_launch<true>(a, w0, w1, out, p, grid, smem, stream)
                : plain::pool2_launch<false>(a, w0, w1, out, p, grid, smem, stream);
  }
  if (p.trace != nullptr) {
    if (is_a4d(v))
      return bf16 ? traced::launch_variant_a4d<true>(v, a, w0, w1, out, p, grid, smem, stream)
                  : traced::launch_variant_a4d<false>(v, a, w0, w1, out, p, grid, smem, stream);
    return bf16 ? traced::launch_variant_a2d<true>(v, a, w0, w1, out, p, grid, smem, stream)
                : traced::launch_variant_a2d<false>(v, a, w0, w1, out, p, grid, smem, stream);
  }
  if (is_a4d(v))
    return bf16 ? plain::launch_variant_a4d<true>(v, a, w0, w1, out, p, grid, smem, stream)
                : plain::launch_variant_a4d<false>(v, a, w0, w1, out, p, grid, smem, stream);
  return bf16 ? plain::launch_variant_a2d<true>(v, a, w0, w1, out, p, grid, smem, stream)
              : plain::launch_variant_a2d<false>(v, a, w0, w1, out, p, grid, smem, stream);
}

cudaError_t cta2_max_clusters(bool bf16, bool trace, size_t smem, int* clusters, bool pool) {
  if (pool) {
    if (trace)
      return bf16 ? traced::pool2_clusters<true>(smem, clusters)
                  : traced::pool2_clusters<false>(smem, clusters);
    return bf16 ? plain::pool2_clusters<true>(smem, clusters)
                : plain::pool2_clusters<false>(smem, clusters);
  }
  if (trace)
    return bf16 ? traced::cta2_clusters<true>(smem, clusters)
                : traced::cta2_clusters<false>(smem, clusters);
  return bf16 ? plain::cta2_clusters<true>(smem, clusters) : plain::cta2_clusters<false>(smem, clusters);
}

// ------------------------------------------------------------------------------------
// max-pool 2x2 / stride 2, floor mode, NHWC; one thread per 8-channel (16-byte) vector.
// ------------------------------------------------------------------------------------
template <bool BF16>
__device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
  if constexpr (BF16) {
    __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a),
                               *reinterpret_cast<__nv_bfloat162*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    __half2 r = __hmax2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

template <bool BF16>
__device__ __forceinline__ uint4 max4(const uint4& a, const uint4& b) {
  return make_uint4(max2<BF16>(a.x, b.x), max2<BF16>(a.y, b.y), max2<BF16>(a.z, b.z),
                    max2<BF16>(a.w, b.w));
}

template <bool BF16>
__global__ void __launch_bounds__(256) maxpool2x2_kernel(const uint4* __restrict__ x,
                                                         uint4* __restrict__ y, int H, int W,
                                                         int Hp, int Wp, int C8, int64_t total) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int c = static_cast<int>(idx % C8);
    int64_t r = idx / C8;
    const int j = static_cast<int>(r % Wp);
    r /= Wp;
    const int i = static_cast<int>(r % Hp);
    const int64_t n = r / Hp;
    const int64_t row0 = ((n * H + 2 * i) * W + 2 * j) * C8 + c;
    const int64_t row1 = row0 + static_cast<int64_t>(W) * C8;
    const uint4 a = __ldg(x + row0), b = __ldg(x + row0 + C8);
    const uint4 d = __ldg(x + row1), e = __ldg(x + row1 + C8);
    y[idx] = max4<BF16>(max4<BF16>(a, b), max4<BF16>(d, e));
  }
}

cudaError_t launch_maxpool(int is_bf16, int N, int H, int W, int C, const void* x, void* y,
                           int num_sms, cudaStream_t stream) {
  const int Hp = H / 2, Wp = W / 2, C8 = C / 8;
  const int64_t total = static_cast<int64_t>(N) * Hp * Wp * C8;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (is_bf16)
    maxpool2x2_kernel<true><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint4*>(y), H, W, Hp, Wp, C8, total);
  else
    maxpool2x2_kernel<false><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint4*>(y), H, W, Hp, Wp, C8, total);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// batch normalisation folded into the preceding operator's weights and bias
// ------------------------------------------------------------------------------------
// One thread per weight element (grid-stride): W'[i] = rnd(W[i] * s[co]) with
// s[co] = gamma[co] / sqrt(var[co] + eps) in fp32, and for i < Co also
// b'[i] = rnd((b[i] - mean[i]) * s[i] + beta[i]).  Element-wise, so W_out may be W and
// b_out may be b.
template <bool BF16>
__device__ __forceinline__ float widen(uint16_t v) {
  if constexpr (BF16) return __bfloat162float(__ushort_as_bfloat16(v));
  else return __half2float(__ushort_as_half(v));
}
template <bool BF16>
__device__ __forceinline__ uint16_t narrow(float v) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  else return __half_as_ushort(__float2half_rn(v));
}

template <bool BF16>
__global__ void __launch_bounds__(256) fold_bn_kernel(
    const uint16_t* __restrict__ Wt, const uint16_t* __restrict__ b, const float* gamma,
    const float* beta, const float* mean, const float* var, float eps, int64_t Co, int64_t K,
    int out_inner, uint16_t* W_out, uint16_t* b_out) {
  const int64_t total = Co * K;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += step) {
    const int64_t co = out_inner ? i % Co : i / K;
    const float s = gamma[co] / sqrtf(var[co] + eps);
    W_out[i] = narrow<BF16>(widen<BF16>(Wt[i]) * s);
    if (i < Co) {
      const float si = gamma[i] / sqrtf(var[i] + eps);
      const float bi = b != nullptr ? widen<BF16>(b[i]) : 0.f;
      b_out[i] = narrow<BF16>((bi - mean[i]) * si + beta[i]);
    }
  }
}

cudaError_t launch_fold_batchnorm(int is_bf16, int64_t Co, int64_t K, int out_inner,
                                  const void* Wt, const void* b, const float* gamma,
                                  const float* beta, const float* mean, const float* var,
                                  float eps, void* W_out, void* b_out, int num_sms,
                                  cudaStream_t stream) {
  const int64_t total = Co * K;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  auto* w = static_cast<const uint16_t*>(Wt);
  auto* bb = static_cast<const uint16_t*>(b);
  auto* wo = static_cast<uint16_t*>(W_out);
  auto* bo = static_cast<uint16_t*>(b_out);
  if (is_bf16)
    fold_bn_kernel<true><<<static_cast<int>(blocks), 256, 0, stream>>>(
        w, bb, gamma, beta, mean, var, eps, Co, K, out_inner, wo, bo);
  else
    fold_bn_kernel<false><<<static_cast<int>(blocks), 256, 0, stream>>>(
        w, bb, gamma, beta, mean, var, eps, Co, K, out_inner, wo, bo);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// timeout probe: a barrier that expects one arrival which never comes
// ------------------------------------------------------------------------------------
__global__ void probe_timeout_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    (void)mbar_wait(b, 0u, limit_ns, nullptr, err, KID_PROBE, SITE_PROBE, 0);
}

cudaError_t launch_probe_timeout(uint64_t limit_ns, uint32_t* err, cudaStream_t stream) {
  probe_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace b2b
