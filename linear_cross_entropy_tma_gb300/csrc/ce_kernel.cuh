// ce_kernel.cuh -- launcher of the standalone row-wise cross-entropy kernel.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace flce {

// Workspace: a 256-byte header (status word at 0, completion counter at 4), then one float4 per row.
constexpr size_t kCeHeaderBytes = 256;
inline size_t ce_workspace_bytes(int64_t B) { return kCeHeaderBytes + static_cast<size_t>(B) * 16u; }

// Element types of the logits.
constexpr int kCeBf16 = 0;
constexpr int kCeF16 = 1;
constexpr int kCeF32 = 2;

// logits [B, V] of type dtype; dlogits: the same buffer (in place), a separate [B, V] buffer of the same
// type, or NULL (loss sums only).  Both buffers start on a 16-byte boundary.
cudaError_t launch_ce_rows(const void* logits, void* dlogits, int dtype, const int64_t* labels, int64_t B, int64_t V,
                           int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum, int64_t* n_valid,
                           void* workspace, int num_sms, cudaStream_t stream);

}  // namespace flce
