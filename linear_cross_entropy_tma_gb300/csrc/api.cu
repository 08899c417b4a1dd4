// api.cu -- the C ABI of libflce.so: argument validation, device checks, tensor-map encoding and
// dispatch to the kernels.  No memory is allocated here; every buffer comes from the caller.
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "../../include/flce.h"
#include "ce_kernel.cuh"
#include "flce_kernels.cuh"
#include "grad_ops.cuh"

namespace {

thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The kernels are built for sm_103a only; anything else cannot run them.
flce_status check_device(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return FLCE_ERR_NO_DEVICE;
  }
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
    set_error("cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    return FLCE_ERR_NO_DEVICE;
  }
  if (major != 10 || minor != 3) {
    set_error("device %d has compute capability %d.%d; libflce.so is built for sm_103a (10.3)", dev, major, minor);
    return FLCE_ERR_NO_DEVICE;
  }
  return FLCE_OK;
}

flce_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return FLCE_OK;
  if (g_last_error[0] == '\0' || e != cudaErrorInvalidValue) set_error("%s: %s", what, cudaGetErrorString(e));
  return FLCE_ERR_CUDA;
}

constexpr int64_t kMax32 = (int64_t(1) << 31) - 1;

}  // namespace

namespace flce {

void set_last_error_message(const char* msg) { set_error("%s", msg); }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, char* err,
                    size_t err_len) {
  static EncodeTiledFn encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || fn == nullptr || q != cudaDriverEntryPointSuccess) {
      snprintf(err, err_len, "cuTensorMapEncodeTiled is not available from the driver");
      return false;
    }
    encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu bf16 tensor, box %u x 64", int(r),
             static_cast<unsigned long long>(rows), static_cast<unsigned long long>(cols), box_rows);
    return false;
  }
  return true;
}

}  // namespace flce

extern "C" {

size_t flce_workspace_size(int64_t BT, int64_t H, int64_t V) {
  if (BT < 0 || H < 0 || V < 0) return 0;
  return flce::fused_workspace_bytes(BT, V);
}

size_t flce_workspace_size_ex(int64_t BT, int64_t H, int64_t V, const flce_fwd_bwd_options* options) {
  if (BT < 0 || H < 0 || V < 0) return 0;
  size_t n = flce::fused_workspace_bytes(BT, V);
  if (options != nullptr && options->sort_vocab != 0) n += flce::vocab_sort_workspace_bytes(BT, H, V);
  return n;
}

static flce_status fwd_bwd_impl(const uint16_t* hidden, const uint16_t* W, const float* bias, const int64_t* target,
                                int64_t BT, int64_t H, int64_t V, int64_t ignore_index, int reduction, float z_loss,
                                float* loss, uint16_t* grad_input, float* grad_W, float* grad_bias, int64_t* n_valid,
                                void* workspace, size_t workspace_bytes, const flce_fwd_bwd_options* options,
                                void* stream, void* const* events, int n_events) {
  g_last_error[0] = '\0';
  const flce_fwd_bwd_options opt =
      options != nullptr ? *options : flce_fwd_bwd_options{1.0f, nullptr, nullptr, 0, nullptr, 0.0f, 0, nullptr, nullptr, 0, 0, 0, 0u};
  if (n_events != 0 && (n_events != 5 || events == nullptr)) {
    set_error("n_events must be 0 or 5 (with a non-NULL event array)");
    return FLCE_ERR_INVALID_ARG;
  }
  if (BT < 0 || H <= 0 || V <= 0) {
    set_error("sizes must satisfy BT >= 0, H > 0, V > 0 (got %lld, %lld, %lld)", (long long)BT, (long long)H,
              (long long)V);
    return FLCE_ERR_INVALID_ARG;
  }
  if (reduction != FLCE_REDUCTION_MEAN && reduction != FLCE_REDUCTION_SUM && reduction != FLCE_REDUCTION_NONE) {
    set_error("reduction must be 0 (mean), 1 (sum) or 2 (none), got %d", reduction);
    return FLCE_ERR_INVALID_ARG;
  }
  if (W == nullptr || workspace == nullptr || (BT > 0 && (hidden == nullptr || target == nullptr)) ||
      (loss == nullptr && reduction != FLCE_REDUCTION_NONE)) {
    set_error("hidden, W, target, loss and workspace must not be NULL (loss may be NULL only for reduction none)");
    return FLCE_ERR_INVALID_ARG;
  }
  if (opt.grad_loss_per_token != nullptr && reduction != FLCE_REDUCTION_NONE) {
    set_error("grad_loss_per_token is only defined for reduction none");
    return FLCE_ERR_INVALID_ARG;
  }
  if (!std::isfinite(opt.grad_scale)) {
    set_error("grad_scale must be finite");
    return FLCE_ERR_INVALID_ARG;
  }
  if (!(opt.filter_eps >= 0.0f) || !std::isfinite(opt.filter_eps)) {
    set_error("filter_eps must be finite and >= 0");
    return FLCE_ERR_INVALID_ARG;
  }
  if (opt.debug_stall_us > 1000000u) {
    set_error("debug_stall_us must be at most 1000000 (1 s), got %u", opt.debug_stall_us);
    return FLCE_ERR_INVALID_ARG;
  }
  if (opt.vocab_splits < 0 || opt.token_splits < 0) {
    set_error("vocab_splits and token_splits must be >= 0, got %d and %d", opt.vocab_splits, opt.token_splits);
    return FLCE_ERR_INVALID_ARG;
  }
  if (opt.sort_vocab == 0 && (opt.logit_avg != nullptr || opt.vocab_order != nullptr)) {
    set_error("logit_avg and vocab_order are outputs of the vocabulary sort (set sort_vocab)");
    return FLCE_ERR_INVALID_ARG;
  }
  if (bias == nullptr && grad_bias != nullptr) {
    set_error("grad_bias requires a bias");
    return FLCE_ERR_INVALID_ARG;
  }
  if ((grad_input != nullptr && (const void*)grad_input == (const void*)hidden) ||
      (grad_W != nullptr && (const void*)grad_W == (const void*)W)) {
    set_error("outputs must not alias the inputs");
    return FLCE_ERR_INVALID_ARG;
  }
  if (H % 8 != 0 || BT > kMax32 || V > kMax32 || H > 65536) {
    set_error("unsupported sizes: need H %% 8 == 0 and H <= 65536, BT and V below 2^31 (got BT=%lld H=%lld V=%lld)",
              (long long)BT, (long long)H, (long long)V);
    return FLCE_ERR_UNSUPPORTED;
  }
  if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(grad_input, 16) || !aligned(grad_W, 16) ||
      !aligned(workspace, 256) || !aligned(bias, 4) || !aligned(grad_bias, 4) || !aligned(loss, 4) ||
      !aligned(target, 8) || !aligned(n_valid, 8) || !aligned(opt.loss_per_token, 4) ||
      !aligned(opt.grad_loss_per_token, 4) || !aligned(opt.entropy, 4) || !aligned(opt.logit_avg, 4) ||
      !aligned(opt.vocab_order, 4)) {
    set_error("misaligned pointer (hidden, W, grad_input, grad_W need 16 bytes; workspace 256)");
    return FLCE_ERR_MISALIGNED;
  }
  const size_t need = flce_workspace_size_ex(BT, H, V, &opt);
  if (workspace_bytes < need) {
    set_error("workspace has %zu bytes, needs %zu", workspace_bytes, need);
    return FLCE_ERR_WORKSPACE_TOO_SMALL;
  }
  int num_sms = 0;
  const flce_status ds = check_device(&num_sms);
  if (ds != FLCE_OK) return ds;

  flce::FusedArgs a{};
  a.hidden = hidden;
  a.W = W;
  a.bias = bias;
  a.target = target;
  a.BT = BT;
  a.H = H;
  a.V = V;
  a.ignore_index = ignore_index;
  a.reduction = reduction;
  a.z_loss = z_loss;
  a.loss = loss;
  a.grad_input = grad_input;
  a.grad_W = grad_W;
  a.grad_bias = grad_bias;
  a.n_valid_out = n_valid;
  a.grad_scale = opt.grad_scale;
  a.grad_tok = opt.grad_loss_per_token;
  a.loss_tok = opt.loss_per_token;
  a.accumulate = opt.accumulate != 0;
  a.entropy = opt.entropy;
  a.filter_eps = opt.filter_eps;
  a.sort_vocab = opt.sort_vocab != 0;
  a.logit_avg_out = opt.logit_avg;
  a.vocab_order_out = opt.vocab_order;
  a.separate_lse = opt.separate_lse_pass != 0;
  a.vocab_splits = opt.vocab_splits;
  a.token_splits = opt.token_splits;
  a.debug_stall_us = opt.debug_stall_us;
  char err[256] = "";
  const cudaError_t e = flce::launch_fused(a, workspace, num_sms, static_cast<cudaStream_t>(stream), err, sizeof(err),
                                           n_events ? reinterpret_cast<cudaEvent_t const*>(events) : nullptr);
  if (e != cudaSuccess && err[0] != '\0') set_error("%s", err);
  return from_cuda(e, "flce_fwd_bwd launch");
}

flce_status flce_fwd_bwd(const uint16_t* hidden, const uint16_t* W, const float* bias, const int64_t* target,
                         int64_t BT, int64_t H, int64_t V, int64_t ignore_index, int reduction, float z_loss,
                         float* loss, uint16_t* grad_input, float* grad_W, float* grad_bias, int64_t* n_valid,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_bwd_impl(hidden, W, bias, target, BT, H, V, ignore_index, reduction == FLCE_REDUCTION_NONE ? -1 : reduction,
                      z_loss, loss, grad_input, grad_W, grad_bias, n_valid, workspace, workspace_bytes, nullptr,
                      stream, nullptr, 0);
}

flce_status flce_fwd_bwd_ex(const uint16_t* hidden, const uint16_t* W, const float* bias, const int64_t* target,
                            int64_t BT, int64_t H, int64_t V, int64_t ignore_index, int reduction, float z_loss,
                            float* loss, uint16_t* grad_input, float* grad_W, float* grad_bias, int64_t* n_valid,
                            void* workspace, size_t workspace_bytes, const flce_fwd_bwd_options* options,
                            void* stream) {
  return fwd_bwd_impl(hidden, W, bias, target, BT, H, V, ignore_index, reduction, z_loss, loss, grad_input, grad_W,
                      grad_bias, n_valid, workspace, workspace_bytes, options, stream, nullptr, 0);
}

flce_status flce_fwd_bwd_timed(const uint16_t* hidden, const uint16_t* W, const float* bias, const int64_t* target,
                               int64_t BT, int64_t H, int64_t V, int64_t ignore_index, int reduction, float z_loss,
                               float* loss, uint16_t* grad_input, float* grad_W, float* grad_bias, int64_t* n_valid,
                               void* workspace, size_t workspace_bytes, void* stream, void* const* events,
                               int n_events) {
  return fwd_bwd_impl(hidden, W, bias, target, BT, H, V, ignore_index, reduction == FLCE_REDUCTION_NONE ? -1 : reduction,
                      z_loss, loss, grad_input, grad_W, grad_bias, n_valid, workspace, workspace_bytes, nullptr,
                      stream, events, n_events);
}

size_t ce_workspace_size(int64_t B, int64_t V) {
  if (B < 0 || V < 0) return 0;
  return flce::ce_workspace_bytes(B);
}

static flce_status ce_impl(const void* logits, void* dlogits, int dtype, const int64_t* labels, int64_t B, int64_t V,
                           int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum, int64_t* n_valid,
                           void* workspace, size_t workspace_bytes, void* stream, const char* name) {
  g_last_error[0] = '\0';
  if (B < 0 || V <= 0) {
    set_error("sizes must satisfy B >= 0, V > 0 (got %lld, %lld)", (long long)B, (long long)V);
    return FLCE_ERR_INVALID_ARG;
  }
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_F16 && dtype != FLCE_DTYPE_F32) {
    set_error("dtype must be FLCE_DTYPE_BF16, FLCE_DTYPE_F16 or FLCE_DTYPE_F32, got %d", dtype);
    return FLCE_ERR_INVALID_ARG;
  }
  if (ce_sum == nullptr || z_sum == nullptr || n_valid == nullptr || workspace == nullptr ||
      (B > 0 && (logits == nullptr || labels == nullptr))) {
    set_error("logits, labels, ce_sum, z_sum, n_valid and workspace must not be NULL");
    return FLCE_ERR_INVALID_ARG;
  }
  if (B > kMax32 || V > kMax32) {
    set_error("unsupported sizes: B and V must be below 2^31");
    return FLCE_ERR_UNSUPPORTED;
  }
  const size_t elem = dtype == FLCE_DTYPE_F32 ? 4u : 2u;
  if (dlogits != nullptr && dlogits != logits) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(dlogits);
    const uintptr_t n = static_cast<uintptr_t>(B) * static_cast<uintptr_t>(V) * elem;
    if (a < b + n && b < a + n) {
      set_error("a separate dlogits buffer must not overlap the logits");
      return FLCE_ERR_INVALID_ARG;
    }
  }
  if (!aligned(logits, 16) || !aligned(dlogits, 16) || !aligned(workspace, 256) || !aligned(labels, 8) ||
      !aligned(ce_sum, 4) || !aligned(z_sum, 4) || !aligned(n_valid, 8)) {
    set_error("misaligned pointer (logits and dlogits need 16 bytes, workspace 256)");
    return FLCE_ERR_MISALIGNED;
  }
  const size_t need = ce_workspace_size(B, V);
  if (workspace_bytes < need) {
    set_error("workspace has %zu bytes, needs %zu", workspace_bytes, need);
    return FLCE_ERR_WORKSPACE_TOO_SMALL;
  }
  int num_sms = 0;
  const flce_status ds = check_device(&num_sms);
  if (ds != FLCE_OK) return ds;
  return from_cuda(flce::launch_ce_rows(logits, dlogits, dtype, labels, B, V, ignore_index, z_loss, ce_sum, z_sum,
                                        n_valid, workspace, num_sms, static_cast<cudaStream_t>(stream)),
                   name);
}

flce_status ce_with_grad(uint16_t* logits, const int64_t* labels, int64_t B, int64_t V, int64_t ignore_index,
                         float z_loss, float* ce_sum, float* z_sum, int64_t* n_valid, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return ce_impl(logits, logits, FLCE_DTYPE_BF16, labels, B, V, ignore_index, z_loss, ce_sum, z_sum, n_valid,
                 workspace, workspace_bytes, stream, "ce_with_grad launch");
}

flce_status ce_with_grad_ex(const void* logits, void* dlogits, int dtype, const int64_t* labels, int64_t B, int64_t V,
                            int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum, int64_t* n_valid,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return ce_impl(logits, dlogits, dtype, labels, B, V, ignore_index, z_loss, ce_sum, z_sum, n_valid, workspace,
                 workspace_bytes, stream, "ce_with_grad_ex launch");
}

flce_status flce_scale_gradient(void* grad, int dtype, int64_t n, const float* upstream, const int64_t* divisor,
                                void* stream) {
  g_last_error[0] = '\0';
  if (dtype != FLCE_DTYPE_BF16 && dtype != FLCE_DTYPE_F16 && dtype != FLCE_DTYPE_F32) {
    set_error("dtype must be FLCE_DTYPE_BF16, FLCE_DTYPE_F16 or FLCE_DTYPE_F32, got %d", dtype);
    return FLCE_ERR_INVALID_ARG;
  }
  if (n < 0 || upstream == nullptr || (n > 0 && grad == nullptr)) {
    set_error("need n >= 0 and non-NULL grad and upstream (got n = %lld)", (long long)n);
    return FLCE_ERR_INVALID_ARG;
  }
  if (!aligned(grad, 16) || !aligned(upstream, 4) || !aligned(divisor, 8)) {
    set_error("misaligned pointer (grad needs 16 bytes, upstream 4, divisor 8)");
    return FLCE_ERR_MISALIGNED;
  }
  int num_sms = 0;
  const flce_status ds = check_device(&num_sms);
  if (ds != FLCE_OK) return ds;
  return from_cuda(flce::launch_scale(grad, n, dtype, upstream, divisor, num_sms, static_cast<cudaStream_t>(stream)),
                   "flce_scale_gradient launch");
}

flce_status ce_reduce_loss(const float* ce_sum, const float* z_sum, const int64_t* n_valid, float z_loss,
                           int reduction, float* loss, void* stream) {
  g_last_error[0] = '\0';
  if (reduction != FLCE_REDUCTION_MEAN && reduction != FLCE_REDUCTION_SUM) {
    set_error("reduction must be 0 (mean) or 1 (sum), got %d", reduction);
    return FLCE_ERR_INVALID_ARG;
  }
  if (ce_sum == nullptr || z_sum == nullptr || n_valid == nullptr || loss == nullptr) {
    set_error("ce_sum, z_sum, n_valid and loss must not be NULL");
    return FLCE_ERR_INVALID_ARG;
  }
  if (!aligned(ce_sum, 4) || !aligned(z_sum, 4) || !aligned(n_valid, 8) || !aligned(loss, 4)) {
    set_error("misaligned pointer (n_valid needs 8 bytes, the others 4)");
    return FLCE_ERR_MISALIGNED;
  }
  int num_sms = 0;
  const flce_status ds = check_device(&num_sms);
  if (ds != FLCE_OK) return ds;
  return from_cuda(flce::launch_ce_reduce_loss(ce_sum, z_sum, n_valid, z_loss, reduction == FLCE_REDUCTION_MEAN, loss,
                                               static_cast<cudaStream_t>(stream)),
                   "ce_reduce_loss launch");
}

flce_status flce_read_device_status(const void* workspace, uint32_t* host_status, void* stream) {
  g_last_error[0] = '\0';
  if (workspace == nullptr || host_status == nullptr) {
    set_error("workspace and host_status must not be NULL");
    return FLCE_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return from_cuda(e, "flce_read_device_status");
}

const char* flce_status_string(flce_status status) {
  switch (status) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG";
    case FLCE_ERR_MISALIGNED: return "FLCE_ERR_MISALIGNED";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "FLCE_ERR_WORKSPACE_TOO_SMALL";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_NO_DEVICE: return "FLCE_ERR_NO_DEVICE";
  }
  return "FLCE_ERR_UNKNOWN";
}

const char* flce_last_error(void) { return g_last_error; }

}  // extern "C"
