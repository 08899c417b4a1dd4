// grad_ops.cuh -- launchers of the loss-reduction and gradient-scaling kernels (grad_ops.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace flce {

// *loss = (*ce_sum + z_loss * *z_sum) / (mean ? max(*n_valid, 1) : 1), one thread.
cudaError_t launch_ce_reduce_loss(const float* ce_sum, const float* z_sum, const int64_t* n_valid, float z_loss,
                                  bool mean, float* loss, cudaStream_t stream);

// buf[0 .. n) *= *upstream / (divisor ? max(*divisor, 1) : 1), in place; buf of element type dtype (the CE
// kernel's codes), 16-byte aligned.
cudaError_t launch_scale(void* buf, int64_t n, int dtype, const float* upstream, const int64_t* divisor, int num_sms,
                         cudaStream_t stream);

}  // namespace flce
