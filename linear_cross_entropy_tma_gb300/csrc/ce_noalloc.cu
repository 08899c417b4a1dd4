// ce_noalloc.cu -- ce_with_grad_noalloc: the standalone CE entry point for callers that cannot
// allocate device memory.
//
// Some callers never get to call cudaMalloc: a plugin inside an inference or training engine whose
// device memory is planned up front and which is handed only its input and output buffers, or a
// service that forbids allocation after start-up because an allocation can block on the allocator
// or fail at run time.  ce_with_grad needs scratch for its per-row partial sums and its completion
// counter; this entry point takes that scratch from a fixed array compiled into the library
// instead of from a caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds
// kNoAllocScratchBytes of device memory for it until the process exits.  Host code cannot use the
// variable's name as a device address (on the host it is only a stand-in symbol), so the first call
// on each device looks the device address up with cudaGetSymbolAddress while that device is current
// and remembers it.  All calls share the one array and it keeps the previous call's contents; the
// launcher clears the part that must start at zero (status word and counter) on every call.  Two
// calls whose kernels overlap on the GPU (different streams, no ordering between them) race on the
// array and give wrong sums.
#include <cstdio>
#include <mutex>

#include "../../include/flce.h"
#include "ce_kernel.cuh"

namespace flce {
void set_last_error_message(const char* msg);  // api.cu: the text flce_last_error() returns
}

namespace {

// header (256 bytes) + 16 bytes per row; the row limit is FLCE_CE_NOALLOC_MAX_ROWS in flce.h
constexpr int64_t kNoAllocMaxRows = FLCE_CE_NOALLOC_MAX_ROWS;
constexpr size_t kNoAllocScratchBytes = flce::kCeHeaderBytes + static_cast<size_t>(kNoAllocMaxRows) * 16u;

static __device__ __align__(256) unsigned char g_ce_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_ce_scratch on `dev` (the current device), looked up once per device.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_ce_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

flce_status ce_with_grad_noalloc(uint16_t* logits, const int64_t* labels, int64_t B, int64_t V, int64_t ignore_index,
                                 float z_loss, float* ce_sum, float* z_sum, int64_t* n_valid, void* stream) {
  char msg[256];
  flce::set_last_error_message("");
  if (B < 0 || V <= 0 || ce_sum == nullptr || z_sum == nullptr || n_valid == nullptr ||
      (B > 0 && (logits == nullptr || labels == nullptr))) {
    snprintf(msg, sizeof(msg), "ce_with_grad_noalloc: need B >= 0 and V > 0 (got %lld, %lld) and non-NULL logits, "
             "labels, ce_sum, z_sum and n_valid", static_cast<long long>(B), static_cast<long long>(V));
    flce::set_last_error_message(msg);
    return FLCE_ERR_INVALID_ARG;
  }
  if (V > (int64_t(1) << 31) - 1) {
    snprintf(msg, sizeof(msg), "ce_with_grad_noalloc: V must be below 2^31 (got %lld)", static_cast<long long>(V));
    flce::set_last_error_message(msg);
    return FLCE_ERR_UNSUPPORTED;
  }
  if (B > kNoAllocMaxRows) {
    snprintf(msg, sizeof(msg),
             "ce_with_grad_noalloc handles at most %lld rows (got %lld); use ce_with_grad with a workspace",
             static_cast<long long>(kNoAllocMaxRows), static_cast<long long>(B));
    flce::set_last_error_message(msg);
    return FLCE_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) != 0 || (reinterpret_cast<uintptr_t>(labels) & 7u) != 0 ||
      (reinterpret_cast<uintptr_t>(ce_sum) & 3u) != 0 || (reinterpret_cast<uintptr_t>(z_sum) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(n_valid) & 7u) != 0) {
    flce::set_last_error_message("ce_with_grad_noalloc: misaligned pointer (logits need 16 bytes, labels and n_valid "
                                 "8, ce_sum and z_sum 4)");
    return FLCE_ERR_MISALIGNED;
  }
  int dev = 0, major = 0, minor = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || major != 10 ||
      minor != 3) {
    (void)cudaGetLastError();
    snprintf(msg, sizeof(msg), "ce_with_grad_noalloc: the current device (%d) is not a compute capability 10.3 GPU "
             "(or the query failed)", dev);
    flce::set_last_error_message(msg);
    return FLCE_ERR_NO_DEVICE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    flce::set_last_error_message(msg);
    return FLCE_ERR_CUDA;
  }
  e = flce::launch_ce_rows(logits, logits, flce::kCeBf16, labels, B, V, ignore_index, z_loss, ce_sum, z_sum, n_valid,
                           scratch, num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "ce_with_grad_noalloc launch: %s", cudaGetErrorString(e));
    flce::set_last_error_message(msg);
    return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

}  // extern "C"
