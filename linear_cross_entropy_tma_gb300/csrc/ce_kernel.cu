// ce_kernel.cu -- standalone row-wise cross-entropy over materialised logits (bf16, fp16 or fp32), with
// the logits gradient written in place or to a separate buffer ("Greyhound -- Cross-Entropy", "Kernel
// design": one block per row, fp32 online max/sum across the row, warp reductions to the row LSE, a
// second pass that overwrites the logits with dlogits; z-loss scales the softmax term before the
// target column is adjusted; "Shape and dtype constraints": bf16, fp16 or fp32 logits).
//
// GB300 shape of it: a persistent grid of two 512-thread CTAs per SM walks the rows.  The first 80 KiB
// of each row (its "head") is fetched into shared memory by one bulk copy, issued as soon as the
// previous row no longer needs the buffer; pass 1 streams the rest of the row with 16-byte loads
// tagged to stay in L2 while the head lands, then reads the head from shared memory; pass 2 writes
// the head's dlogits from shared memory and re-reads the rest (an L2 hit: about 2 x 152 x 170 KB
// = 52 MB of rows are in flight at bf16), storing with 16-byte stores tagged evict-first.  HBM
// therefore sees one read and one write of the logits.  Without a gradient buffer pass 2 is skipped.
// Per-row (ce, LSE^2, valid) land in the workspace; the last CTA to finish sums them in a fixed
// order (float64), so the three outputs are deterministic.
#include <cuda_fp16.h>

#include "ce_kernel.cuh"
#include "sm100.cuh"

namespace flce {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCtasPerSm = 2;
// The first kCacheVec 16-byte vectors of each row are kept in shared memory between the two passes
// (80 KiB per CTA), so only the rest of the row is read a second time.
constexpr int kCacheVec = 5120;
constexpr size_t kCacheBytes = static_cast<size_t>(kCacheVec) * 16u;
constexpr int kUnroll = 4;  // 16-byte vectors per thread in flight per step

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld16_hint(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void st16_hint(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
               ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// Merge two (max, sum) pairs of the online softmax; max values are in the log2 domain.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  const float a = (m == mn) ? s : s * ex2_approx(m - mn);
  const float b = (m2 == mn) ? s2 : s2 * ex2_approx(m2 - mn);
  m = mn;
  s = a + b;
}

// Element types of the logits: raw storage, elements per 16-byte vector, and conversions.
struct Bf16Elem {
  using raw = uint16_t;
  static constexpr int kPer = 8;
  __device__ static float load1(raw r) { return __uint_as_float(static_cast<uint32_t>(r) << 16); }
  __device__ static raw store1(float f) { return static_cast<uint16_t>(pack_bf16x2(f, 0.0f) & 0xFFFFu); }
  __device__ static void unpack(const uint4 v, float (&x)[kPer]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_lo(w[i]);
      x[2 * i + 1] = bf16_hi(w[i]);
    }
  }
  __device__ static uint4 pack(const float (&g)[kPer]) {
    return make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]),
                      pack_bf16x2(g[6], g[7]));
  }
};

struct F16Elem {
  using raw = uint16_t;
  static constexpr int kPer = 8;
  __device__ static float load1(raw r) { return __half2float(__ushort_as_half(r)); }
  __device__ static raw store1(float f) { return __half_as_ushort(__float2half_rn(f)); }
  __device__ static void unpack(const uint4 v, float (&x)[kPer]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ static uint4 pack(const float (&g)[kPer]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(g[2 * i], g[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

struct F32Elem {
  using raw = float;
  static constexpr int kPer = 4;
  __device__ static float load1(raw r) { return r; }
  __device__ static raw store1(float f) { return f; }
  __device__ static void unpack(const uint4 v, float (&x)[kPer]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 pack(const float (&g)[kPer]) {
    return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]), __float_as_uint(g[3]));
  }
};

template <class E>
__device__ __forceinline__ void accumulate_vec(const uint4 v, float& m, float& s) {
  float x[E::kPer];
  E::unpack(v, x);
  float cm = x[0];
#pragma unroll
  for (int i = 1; i < E::kPer; ++i) cm = fmaxf(cm, x[i]);
  const float mn = fmaxf(m, cm * kLog2e);
  float acc = s * ex2_approx(m - mn);  // m = -inf on the first call gives 0 * 0
#pragma unroll
  for (int i = 0; i < E::kPer; ++i) acc += ex2_approx(fmaf(x[i], kLog2e, -mn));
  m = mn;
  s = acc;
}

// dlogits of one 16-byte vector of consecutive columns starting at column c0 (softmax * zf - onehot).
template <class E>
__device__ __forceinline__ uint4 grad_vec(const uint4 v, int64_t c0, int64_t y, float lse2, float zf) {
  float g[E::kPer];
  E::unpack(v, g);
#pragma unroll
  for (int i = 0; i < E::kPer; ++i) g[i] = ex2_approx(fmaf(g[i], kLog2e, -lse2)) * zf;
  const uint64_t t = static_cast<uint64_t>(y - c0);  // target column relative to c0
  if (t < static_cast<uint64_t>(E::kPer)) {
#pragma unroll
    for (int i = 0; i < E::kPer; ++i)
      if (static_cast<uint64_t>(i) == t) g[i] -= 1.0f;
  }
  return E::pack(g);
}

template <class E>
__device__ __forceinline__ float grad1(typename E::raw raw, int64_t c, int64_t y, float lse2, float zf) {
  const float g = ex2_approx(fmaf(E::load1(raw), kLog2e, -lse2)) * zf;
  return (c == y) ? g - 1.0f : g;
}

// in: logits [B, V]; out: dlogits [B, V] (== in for the in-place call, NULL for no gradient).
template <class E>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
ce_rows_kernel(const typename E::raw* in, typename E::raw* out, const int64_t* __restrict__ labels, int64_t B,
               int64_t V, int64_t ignore_index, float z_loss, float4* __restrict__ row_out,
               uint32_t* __restrict__ status, uint32_t* __restrict__ done_counter, float* __restrict__ ce_sum,
               float* __restrict__ z_sum, int64_t* __restrict__ n_valid) {
  using raw = typename E::raw;
  constexpr int kPer = E::kPer;
  constexpr int kShift = sizeof(raw) == 2 ? 1 : 2;
  extern __shared__ uint4 s_cache[];  // kCacheVec vectors of the current row
  __shared__ uint64_t s_head_bar;
  __shared__ float s_m[kWarps], s_s[kWarps];
  __shared__ float s_lse2;
  __shared__ float s_zy;
  __shared__ double s_red[2][kWarps];
  __shared__ long long s_cnt[kWarps];
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const bool want_grad = (out != nullptr);
  const uint64_t keep = policy_evict_last();
  const uint64_t drop = policy_evict_first();

  // Head of row r: the first min(kCacheVec, nvec) 16-byte vectors of its aligned part.
  auto head_bytes = [&](int64_t r, const uint4*& src) -> uint32_t {
    const int64_t y = labels[r];
    if (!((y != ignore_index) && (y >= 0) && (y < V))) return 0u;
    const raw* rw = in + r * V;
    const uintptr_t a = reinterpret_cast<uintptr_t>(rw);
    const int64_t hd_raw = static_cast<int64_t>(((16u - (a & 15u)) & 15u) >> kShift);
    const int64_t hd = hd_raw < V ? hd_raw : V;
    const int64_t nv = (V - hd) / kPer;
    src = reinterpret_cast<const uint4*>(rw + hd);
    return static_cast<uint32_t>((nv < kCacheVec ? nv : kCacheVec) * 16);
  };
  auto prefetch_head = [&](int64_t r) {
    const uint4* src = nullptr;
    const uint32_t bytes = head_bytes(r, src);
    if (bytes) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&s_head_bar, bytes);
      bulk_load_1d_hint(s_cache, src, bytes, &s_head_bar, keep);
    }
  };
  if (tid == 0) {
    mbar_init(&s_head_bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  uint32_t head_phase = 0;
  volatile int no_abort = 0;
  if (tid == 0 && blockIdx.x < B) prefetch_head(blockIdx.x);

  for (int64_t r = blockIdx.x; r < B; r += gridDim.x) {
    const int64_t y = labels[r];
    const bool valid = (y != ignore_index) && (y >= 0) && (y < V);
    const raw* row = in + r * V;
    raw* orow = want_grad ? out + r * V : nullptr;
    // 16-byte aligned middle part of the row; scalar head and tail around it (in and out rows have
    // the same alignment: both buffers start on a 16-byte boundary)
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    const int64_t head_raw = static_cast<int64_t>(((16u - (addr & 15u)) & 15u) >> kShift);
    const int64_t head = head_raw < V ? head_raw : V;
    const int64_t nvec = (V - head) / kPer;
    const int64_t tail0 = head + nvec * kPer;
    const uint4* vrow = reinterpret_cast<const uint4*>(row + head);
    uint4* ovrow = want_grad ? reinterpret_cast<uint4*>(orow + head) : nullptr;

    if (!valid) {
      if (tid == 0) {
        if (y != ignore_index) atomicOr(status, kStatusBadTarget);
        row_out[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        // no head was fetched for this row; fetch the next row's head now
        if (r + gridDim.x < B) prefetch_head(r + gridDim.x);
      }
      if (want_grad) {
        for (int64_t i = tid; i < nvec; i += kThreads) st16_hint(ovrow + i, make_uint4(0, 0, 0, 0), drop);
        for (int64_t c = tid; c < head; c += kThreads) orow[c] = E::store1(0.f);
        for (int64_t c = tail0 + tid; c < V; c += kThreads) orow[c] = E::store1(0.f);
      }
      continue;
    }

    if (tid == 0) s_zy = E::load1(row[y]);

    // ---- pass 1: online (max, sum) in the log2 domain
    float m = -INFINITY, s = 0.f;
    for (int64_t c = tid; c < head; c += kThreads) merge_ms(m, s, E::load1(row[c]) * kLog2e, 1.0f);
    for (int64_t c = tail0 + tid; c < V; c += kThreads) merge_ms(m, s, E::load1(row[c]) * kLog2e, 1.0f);
    const int64_t ncache = nvec < kCacheVec ? nvec : kCacheVec;
    // the tail (vectors ncache..nvec-1) from global memory while the head's bulk copy lands
    int64_t i = ncache + tid;
    for (; i + (kUnroll - 1) * kThreads < nvec; i += kUnroll * kThreads) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = ld16_hint(vrow + i + u * kThreads, keep);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) accumulate_vec<E>(v[u], m, s);
    }
    for (; i < nvec; i += kThreads) accumulate_vec<E>(ld16_hint(vrow + i, keep), m, s);
    // the head from shared memory
    if (ncache > 0) {
      if (!mbar_wait(&s_head_bar, head_phase, &no_abort) && (tid & 31) == 0) atomicOr(status, kStatusTimeout);
      head_phase ^= 1u;
      for (int64_t k = tid; k < ncache; k += kThreads) accumulate_vec<E>(s_cache[k], m, s);
    }

#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
      merge_ms(m, s, m2, s2);
    }
    if ((tid & 31) == 0) {
      s_m[warp] = m;
      s_s[warp] = s;
    }
    __syncthreads();
    if (warp == 0) {
      m = (tid < kWarps) ? s_m[tid] : -INFINITY;
      s = (tid < kWarps) ? s_s[tid] : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        merge_ms(m, s, m2, s2);
      }
      if (tid == 0) {
        const float lse2 = m + __log2f(s);
        s_lse2 = lse2;
        const float lse = lse2 * kLn2;
        row_out[r] = make_float4(lse - s_zy, lse * lse, 1.f, 0.f);
        // without a gradient the cache is free as soon as every thread has read it (the barrier above)
        if (!want_grad && r + gridDim.x < B) prefetch_head(r + gridDim.x);
      }
    }
    __syncthreads();
    if (!want_grad) continue;
    const float lse2 = s_lse2;
    const float zf = 1.0f + 2.0f * z_loss * (lse2 * kLn2);

    // ---- pass 2: dlogits
    for (int64_t c = tid; c < head; c += kThreads) orow[c] = E::store1(grad1<E>(row[c], c, y, lse2, zf));
    for (int64_t c = tail0 + tid; c < V; c += kThreads) orow[c] = E::store1(grad1<E>(row[c], c, y, lse2, zf));
    for (int64_t k = tid; k < ncache; k += kThreads)
      st16_hint(ovrow + k, grad_vec<E>(s_cache[k], head + k * kPer, y, lse2, zf), drop);
    // every thread is done reading the cache: start copying the head of this CTA's next row
    __syncthreads();
    if (tid == 0 && r + gridDim.x < B) prefetch_head(r + gridDim.x);
    i = ncache + tid;
    for (; i + (kUnroll - 1) * kThreads < nvec; i += kUnroll * kThreads) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = ld16_hint(vrow + i + u * kThreads, drop);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        st16_hint(ovrow + i + u * kThreads, grad_vec<E>(v[u], head + (i + u * kThreads) * kPer, y, lse2, zf), drop);
    }
    for (; i < nvec; i += kThreads)
      st16_hint(ovrow + i, grad_vec<E>(ld16_hint(vrow + i, drop), head + i * kPer, y, lse2, zf), drop);
    __syncthreads();  // s_m / s_s / s_lse2 / s_zy are reused by the next row
  }

  // ---- the last CTA to finish reduces the per-row terms in row order
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(done_counter, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  double ce = 0.0, zz = 0.0;
  long long cnt = 0;
  for (int64_t k = tid; k < B; k += kThreads) {
    const float4 v = __ldcg(row_out + k);
    ce += v.x;
    zz += v.y;
    cnt += (v.z != 0.f) ? 1 : 0;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ce += __shfl_xor_sync(0xffffffffu, ce, off);
    zz += __shfl_xor_sync(0xffffffffu, zz, off);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  }
  if ((tid & 31) == 0) {
    s_red[0][warp] = ce;
    s_red[1][warp] = zz;
    s_cnt[warp] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    double a = 0.0, b = 0.0;
    long long n = 0;
    for (int w = 0; w < kWarps; ++w) {
      a += s_red[0][w];
      b += s_red[1][w];
      n += s_cnt[w];
    }
    *ce_sum = static_cast<float>(a);
    *z_sum = static_cast<float>(b);
    *n_valid = n;
    *done_counter = 0u;
  }
}


template <class E>
cudaError_t launch_ce_rows_t(const void* logits, void* dlogits, const int64_t* labels, int64_t B, int64_t V,
                             int64_t ignore_index, float z_loss, float4* row_out, uint32_t* status, uint32_t* counter,
                             float* ce_sum, float* z_sum, int64_t* n_valid, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(ce_rows_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kCacheBytes));
  if (e != cudaSuccess) return e;
  const int64_t cap = static_cast<int64_t>(num_sms) * kCtasPerSm;
  const int64_t grid = B < cap ? B : cap;
  using raw = typename E::raw;
  ce_rows_kernel<E><<<static_cast<unsigned>(grid), kThreads, kCacheBytes, stream>>>(
      static_cast<const raw*>(logits), static_cast<raw*>(dlogits), labels, B, V, ignore_index, z_loss, row_out, status,
      counter, ce_sum, z_sum, n_valid);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ce_rows(const void* logits, void* dlogits, int dtype, const int64_t* labels, int64_t B, int64_t V,
                           int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum, int64_t* n_valid,
                           void* workspace, int num_sms, cudaStream_t stream) {
  auto* ws = static_cast<unsigned char*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint32_t* counter = reinterpret_cast<uint32_t*>(ws + 4);
  float4* row_out = reinterpret_cast<float4*>(ws + kCeHeaderBytes);
  cudaError_t e = cudaMemsetAsync(ws, 0, kCeHeaderBytes, stream);
  if (e != cudaSuccess) return e;
  if (B == 0) {
    if ((e = cudaMemsetAsync(ce_sum, 0, sizeof(float), stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(z_sum, 0, sizeof(float), stream)) != cudaSuccess) return e;
    return cudaMemsetAsync(n_valid, 0, sizeof(int64_t), stream);
  }
  switch (dtype) {
    case kCeBf16:
      return launch_ce_rows_t<Bf16Elem>(logits, dlogits, labels, B, V, ignore_index, z_loss, row_out, status, counter,
                                        ce_sum, z_sum, n_valid, num_sms, stream);
    case kCeF16:
      return launch_ce_rows_t<F16Elem>(logits, dlogits, labels, B, V, ignore_index, z_loss, row_out, status, counter,
                                       ce_sum, z_sum, n_valid, num_sms, stream);
    case kCeF32:
      return launch_ce_rows_t<F32Elem>(logits, dlogits, labels, B, V, ignore_index, z_loss, row_out, status, counter,
                                       ce_sum, z_sum, n_valid, num_sms, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace flce
