// grad_ops.cu -- the two small kernels behind the autograd form of the calls, so that a framework's
// backward pass needs no host synchronisation and no arithmetic outside the library:
//   * ce_reduce_loss_kernel: the reduced loss of the standalone CE from its device sums,
//       loss = (ce_sum + z_loss z_sum) / max(n_valid, 1)   (mean; "Greyhound -- Cross-Entropy", "Usage":
//       ce_sum over the clamped valid count)      or   ce_sum + z_loss z_sum   (sum);
//   * scale_kernel: a gradient buffer multiplied in place by the upstream gradient g (a device scalar),
//       optionally divided by max(n, 1) for a device count n -- the d_out factor of "Cut Cross Entropy
//       visualized", "Breakdown: Backward Pass", step 4.
// The scaling kernel is HBM-bound: 16-byte loads and stores, four in flight per thread, a grid-stride loop
// over a grid of a few CTAs per SM; when the factor is exactly 1 it returns without touching the buffer.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ce_kernel.cuh"
#include "grad_ops.cuh"

namespace flce {

namespace {

__global__ void ce_reduce_loss_kernel(const float* __restrict__ ce_sum, const float* __restrict__ z_sum,
                                      const int64_t* __restrict__ n_valid, float z_loss, int mean,
                                      float* __restrict__ loss) {
  float l = *ce_sum;
  if (z_loss != 0.f) l = fmaf(z_loss, *z_sum, l);
  if (mean) l /= static_cast<float>(*n_valid > 1 ? *n_valid : 1);
  *loss = l;
}

__device__ __forceinline__ float scale_factor(const float* upstream, const int64_t* divisor) {
  float g = *upstream;
  if (divisor != nullptr) g /= static_cast<float>(*divisor > 1 ? *divisor : 1);
  return g;
}

// 8 bf16 / fp16 values or 4 fp32 values per 16-byte vector
__device__ __forceinline__ uint4 scale_vec(uint4 v, float g, int dtype) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if (dtype == kCeF32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * g);
  } else if (dtype == kCeBf16) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * g, f.y * g);
      w[k] = *reinterpret_cast<const uint32_t*>(&r);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
      const __half2 r = __floats2half2_rn(f.x * g, f.y * g);
      w[k] = *reinterpret_cast<const uint32_t*>(&r);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void scale_one(void* buf, int64_t i, float g, int dtype) {
  if (dtype == kCeF32) {
    float* p = static_cast<float*>(buf) + i;
    *p *= g;
  } else if (dtype == kCeBf16) {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(buf) + i;
    *p = __float2bfloat16_rn(__bfloat162float(*p) * g);
  } else {
    __half* p = static_cast<__half*>(buf) + i;
    *p = __float2half_rn(__half2float(*p) * g);
  }
}

constexpr int kScaleThreads = 512;
constexpr int kScaleUnroll = 4;

__global__ void __launch_bounds__(kScaleThreads) scale_kernel(void* __restrict__ buf, int64_t n, int dtype,
                                                              const float* __restrict__ upstream,
                                                              const int64_t* __restrict__ divisor) {
  const float g = scale_factor(upstream, divisor);
  if (g == 1.0f) return;
  const int per_vec = dtype == kCeF32 ? 4 : 8;
  const int64_t nvec = n / per_vec;
  uint4* v = static_cast<uint4*>(buf);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kScaleUnroll - 1) * stride < nvec; i += kScaleUnroll * stride) {
    uint4 x[kScaleUnroll];
#pragma unroll
    for (int u = 0; u < kScaleUnroll; ++u) x[u] = v[i + u * stride];
#pragma unroll
    for (int u = 0; u < kScaleUnroll; ++u) v[i + u * stride] = scale_vec(x[u], g, dtype);
  }
  for (; i < nvec; i += stride) v[i] = scale_vec(v[i], g, dtype);
  // the elements past the last whole vector
  const int64_t t = nvec * per_vec + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t < n) scale_one(buf, t, g, dtype);
}

}  // namespace

cudaError_t launch_ce_reduce_loss(const float* ce_sum, const float* z_sum, const int64_t* n_valid, float z_loss,
                                  bool mean, float* loss, cudaStream_t stream) {
  ce_reduce_loss_kernel<<<1, 1, 0, stream>>>(ce_sum, z_sum, n_valid, z_loss, mean ? 1 : 0, loss);
  return cudaGetLastError();
}

cudaError_t launch_scale(void* buf, int64_t n, int dtype, const float* upstream, const int64_t* divisor, int num_sms,
                         cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int per_vec = dtype == kCeF32 ? 4 : 8;
  const int64_t nvec = n / per_vec;
  const int64_t want = (nvec + kScaleThreads * kScaleUnroll - 1) / (kScaleThreads * kScaleUnroll);
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 4 * static_cast<int64_t>(num_sms))));
  scale_kernel<<<blocks, kScaleThreads, 0, stream>>>(buf, n, dtype, upstream, divisor);
  return cudaGetLastError();
}

}  // namespace flce
