// vocab_sort.cu -- the vocabulary sort that precedes gradient filtering ("Cut Cross Entropy visualized",
// "Forward pass": logit_avg, the mean logit of each vocabulary entry over the batch; "Vocabulary
// Sorting": the vocabulary ordered by it, so that the entries with large gradients gather in few blocks
// and the rest form long runs of blocks the filter can skip).
//
// GB300 form of the step:
//   * logit_avg[n] = (1/BT) sum_t z[t, n] = W[n] . hbar + b[n] with hbar = (1/BT) sum_t hidden[t] (the sum
//     over tokens commutes with the dot product), so it costs one read of hidden and one of W (two
//     HBM-bound kernels) instead of column sums inside every logits tile of the LSE pass;
//   * a stable least-significant-digit radix sort of the V keys (4 passes of 8 bits: per-block digit
//     histograms, one scan, a stable per-block scatter), largest key first, equal keys by index;
//   * the fused passes then run on a gathered copy of W, the bias and the targets in sorted order; the
//     grad_W pass writes its rows back through the permutation.
#include "flce_kernels.cuh"
#include "sm100.cuh"

namespace flce {

namespace {

constexpr int kColSplits = 64;        // row splits of the hidden column sum
constexpr int kSortThreads = 1024;
constexpr int kSortChunk = 2 * kSortThreads;   // keys per block of the radix passes

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }

// Radix key of a float for a descending sort: larger floats give smaller keys; -0 and +0 are equal.
__device__ __forceinline__ uint32_t descending_key(float x) {
  uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
  const uint32_t ascending = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~ascending;
}

// part[split][k] = sum of hidden[t][k] over this split's rows.  Block: 8 warps over a 256-column strip,
// each lane 8 consecutive columns (one 16-byte load per row).
__global__ void __launch_bounds__(256) hidden_colsum_kernel(const uint16_t* __restrict__ hidden, int BT, int H,
                                                            float* __restrict__ part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 256 + lane * 8;
  const int split = blockIdx.y;
  const int rows_per = (BT + kColSplits - 1) / kColSplits;
  const int r_begin = split * rows_per;
  const int r_end = min(BT, r_begin + rows_per);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c0 < H) {
    // four rows per warp in flight, accumulated in row order
    for (int r = r_begin + warp; r < r_end; r += 32) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = r + 8 * u < r_end ? *reinterpret_cast<const uint4*>(hidden + static_cast<size_t>(r + 8 * u) * H + c0)
                                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] += bf16_to_f32(static_cast<uint16_t>(w[e] & 0xFFFFu));
          acc[2 * e + 1] += bf16_to_f32(static_cast<uint16_t>(w[e] >> 16));
        }
      }
    }
  }
  __shared__ float red[8][256];
#pragma unroll
  for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[e];
  __syncthreads();
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c < H) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w][threadIdx.x];
    part[static_cast<size_t>(split) * H + c] = s;
  }
}

// hbar[k] = (sum over splits in order) / BT (0 for an empty batch).
__global__ void hidden_mean_kernel(const float* __restrict__ part, int BT, int H, float* __restrict__ hbar) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  float s = 0.f;
  for (int i = 0; i < kColSplits; ++i) s += part[static_cast<size_t>(i) * H + c];
  hbar[c] = BT > 0 ? s / static_cast<float>(BT) : 0.f;
}

// avg[n] = W[n] . hbar + b[n]; keys / vals: the first radix input (descending key, index).  One warp per
// vocabulary row; hbar (4 H bytes) is read through the L1 cache.
__global__ void __launch_bounds__(256) logit_avg_kernel(const uint16_t* __restrict__ W, const float* __restrict__ bias,
                                                        const float* __restrict__ hbar, int V, int H,
                                                        float* __restrict__ avg, uint32_t* __restrict__ keys,
                                                        int32_t* __restrict__ vals) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int n = blockIdx.x * warps + warp; n < V; n += gridDim.x * warps) {
    const uint16_t* row = W + static_cast<size_t>(n) * H;
    float s = 0.f;
    // four 16-byte pieces of the row per lane in flight
    for (int c = lane * 8; c < H; c += 1024) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = c + 256 * u < H ? *reinterpret_cast<const uint4*>(row + c + 256 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c + 256 * u >= H) break;
        const float4 h0 = __ldg(reinterpret_cast<const float4*>(hbar + c + 256 * u));
        const float4 h1 = __ldg(reinterpret_cast<const float4*>(hbar + c + 256 * u + 4));
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        const float hb[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s = fmaf(bf16_to_f32(static_cast<uint16_t>(w[e] & 0xFFFFu)), hb[2 * e], s);
          s = fmaf(bf16_to_f32(static_cast<uint16_t>(w[e] >> 16)), hb[2 * e + 1], s);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      const float a = s + (bias != nullptr ? bias[n] : 0.f);
      avg[n] = a;
      keys[n] = descending_key(a);
      vals[n] = n;
    }
  }
}

// hist[b][d]: how many keys of block b's chunk have digit d at `shift`.
__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(const uint32_t* __restrict__ keys, int n, int shift,
                                                                  uint32_t* __restrict__ hist) {
  __shared__ uint32_t h[256];
  if (threadIdx.x < 256) h[threadIdx.x] = 0;
  __syncthreads();
  const int begin = blockIdx.x * kSortChunk;
  const int end = min(n, begin + kSortChunk);
  for (int i = begin + threadIdx.x; i < end; i += kSortThreads) atomicAdd(&h[(keys[i] >> shift) & 0xFFu], 1u);
  __syncthreads();
  if (threadIdx.x < 256) hist[static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x] = h[threadIdx.x];
}

// In place: hist[b][d] becomes the output position of block b's first key with digit d (digits in
// increasing order, blocks in order within a digit).  One block of 256 threads (one per digit).
__global__ void __launch_bounds__(256) radix_scan_kernel(uint32_t* __restrict__ hist, int nb) {
  __shared__ uint32_t tot[256];
  const int d = threadIdx.x;
  uint32_t s = 0;
  for (int b = 0; b < nb; ++b) s += hist[static_cast<size_t>(b) * 256 + d];
  tot[d] = s;
  __syncthreads();
  // exclusive scan over the 256 digit totals (Hillis-Steele in shared memory)
  for (int o = 1; o < 256; o <<= 1) {
    const uint32_t v = d >= o ? tot[d - o] : 0u;
    __syncthreads();
    tot[d] += v;
    __syncthreads();
  }
  uint32_t base = tot[d] - s;
  for (int b = 0; b < nb; ++b) {
    const uint32_t c = hist[static_cast<size_t>(b) * 256 + d];
    hist[static_cast<size_t>(b) * 256 + d] = base;
    base += c;
  }
}

// Stable scatter of block b's chunk: sub-tiles of 1024 keys in index order; within a sub-tile a key's
// place among equal digits is (keys with that digit in earlier warps) + (earlier lanes of its warp).
__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(const uint32_t* __restrict__ keys_in,
                                                                     const int32_t* __restrict__ vals_in, int n,
                                                                     int shift, const uint32_t* __restrict__ offsets,
                                                                     uint32_t* __restrict__ keys_out,
                                                                     int32_t* __restrict__ vals_out) {
  __shared__ uint32_t running[256];   // output position of the next key with each digit
  __shared__ uint32_t total[256];     // keys with each digit in the current sub-tile
  __shared__ uint16_t wcnt[32][256];  // keys with each digit per warp of the current sub-tile
  __shared__ uint16_t wpre[32][256];  // exclusive prefix of wcnt over the warps
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < 256) running[tid] = offsets[static_cast<size_t>(blockIdx.x) * 256 + tid];
  for (int i = tid; i < 32 * 256; i += kSortThreads) wcnt[i >> 8][i & 255] = 0;
  __syncthreads();
  const int begin = blockIdx.x * kSortChunk;
  const int end = min(n, begin + kSortChunk);
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int t0 = begin; t0 < end; t0 += kSortThreads) {
    const int i = t0 + tid;
    const bool valid = i < end;
    const uint32_t key = valid ? keys_in[i] : 0u;
    const int32_t val = valid ? vals_in[i] : 0;
    const uint32_t d = valid ? ((key >> shift) & 0xFFu) : 256u;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const uint32_t rank = __popc(peers & lt_mask);
    if (valid && rank == 0) wcnt[warp][d] = static_cast<uint16_t>(__popc(peers));
    __syncthreads();
    if (tid < 256) {
      uint32_t run = 0;
      for (int w = 0; w < 32; ++w) {
        const uint32_t c = wcnt[w][tid];
        wpre[w][tid] = static_cast<uint16_t>(run);
        wcnt[w][tid] = 0;
        run += c;
      }
      total[tid] = run;
    }
    __syncthreads();
    if (valid) {
      const uint32_t pos = running[d] + wpre[warp][d] + rank;
      keys_out[pos] = key;
      vals_out[pos] = val;
    }
    __syncthreads();
    if (tid < 256) running[tid] += total[tid];
    __syncthreads();
  }
}

// Sorted copies: W_s[i] = W[perm[i]], b_s[i] = b[perm[i]], inv[perm[i]] = i.  One warp per sorted row,
// 16-byte copies (H is a multiple of 8).
__global__ void __launch_bounds__(256) vocab_gather_kernel(const uint16_t* __restrict__ W, const float* __restrict__ bias,
                                                           const int32_t* __restrict__ perm, int V, int H,
                                                           uint16_t* __restrict__ W_s, float* __restrict__ bias_s,
                                                           int32_t* __restrict__ inv, uint32_t* __restrict__ status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  for (int i = blockIdx.x * warps + warp; i < V; i += gridDim.x * warps) {
    const int src = perm[i];
    if (src < 0 || src >= V) {
      // not a permutation: a defect of the sort, reported instead of reading out of bounds
      if (lane == 0) atomicOr(status, kStatusInternal);
      continue;
    }
    const uint4* from = reinterpret_cast<const uint4*>(W + static_cast<size_t>(src) * H);
    uint4* to = reinterpret_cast<uint4*>(W_s + static_cast<size_t>(i) * H);
    const int n16 = H / 8;
    for (int c = lane; c < n16; c += 128) {
      uint4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < n16) t[u] = from[c + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c + 32 * u < n16) to[c + 32 * u] = t[u];
    }
    if (lane == 0) {
      if (bias != nullptr) bias_s[i] = bias[src];
      inv[src] = i;
    }
  }
}

// Targets in sorted vocabulary indices.  Ignored rows and targets outside [0, V) become -1 (the ignore
// index of the sorted call); the latter also set the bad-target status bit here.
__global__ void target_remap_kernel(const int64_t* __restrict__ target, int BT, int V, int64_t ignore_index,
                                    const int32_t* __restrict__ inv, int64_t* __restrict__ out,
                                    uint32_t* __restrict__ status) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= BT) return;
  const int64_t y = target[t];
  if (y == ignore_index) {
    out[t] = -1;
  } else if (y < 0 || y >= V) {
    out[t] = -1;
    atomicOr(status, kStatusBadTarget);
  } else {
    out[t] = inv[y];
  }
}

}  // namespace

size_t vocab_sort_workspace_bytes(int64_t BT, int64_t H, int64_t V) {
  const size_t v = static_cast<size_t>(V > 0 ? V : 0);
  const size_t nb = (v + kSortChunk - 1) / kSortChunk;
  size_t off = 0;
  off += round_up(sizeof(float) * kColSplits * static_cast<size_t>(H), 256);   // column-sum partials
  off += round_up(sizeof(float) * static_cast<size_t>(H), 256);               // hbar
  off += round_up(sizeof(float) * v, 256);                                     // logit_avg
  off += 2 * round_up(sizeof(uint32_t) * v, 256);                              // keys (double buffer)
  off += 2 * round_up(sizeof(int32_t) * v, 256);                               // values (double buffer)
  off += round_up(sizeof(uint32_t) * 256 * nb, 256);                           // block histograms
  off += round_up(sizeof(int32_t) * v, 256);                                   // inverse permutation
  off += round_up(sizeof(float) * v, 256);                                     // sorted bias
  off += round_up(sizeof(int64_t) * static_cast<size_t>(BT > 0 ? BT : 0), 256);  // sorted targets
  off += round_up(sizeof(uint16_t) * v * static_cast<size_t>(H), 256);         // sorted W
  return off;
}

VocabSortWorkspace carve_vocab_sort(void* base, int64_t BT, int64_t H, int64_t V) {
  const size_t v = static_cast<size_t>(V > 0 ? V : 0);
  const size_t nb = (v + kSortChunk - 1) / kSortChunk;
  auto* p = static_cast<unsigned char*>(base);
  VocabSortWorkspace w;
  size_t off = 0;
  w.col_part = reinterpret_cast<float*>(p + off);
  off += round_up(sizeof(float) * kColSplits * static_cast<size_t>(H), 256);
  w.hbar = reinterpret_cast<float*>(p + off);
  off += round_up(sizeof(float) * static_cast<size_t>(H), 256);
  w.logit_avg = reinterpret_cast<float*>(p + off);
  off += round_up(sizeof(float) * v, 256);
  w.keys[0] = reinterpret_cast<uint32_t*>(p + off);
  off += round_up(sizeof(uint32_t) * v, 256);
  w.keys[1] = reinterpret_cast<uint32_t*>(p + off);
  off += round_up(sizeof(uint32_t) * v, 256);
  w.vals[0] = reinterpret_cast<int32_t*>(p + off);
  off += round_up(sizeof(int32_t) * v, 256);
  w.vals[1] = reinterpret_cast<int32_t*>(p + off);
  off += round_up(sizeof(int32_t) * v, 256);
  w.hist = reinterpret_cast<uint32_t*>(p + off);
  off += round_up(sizeof(uint32_t) * 256 * nb, 256);
  w.inv = reinterpret_cast<int32_t*>(p + off);
  off += round_up(sizeof(int32_t) * v, 256);
  w.bias = reinterpret_cast<float*>(p + off);
  off += round_up(sizeof(float) * v, 256);
  w.target = reinterpret_cast<int64_t*>(p + off);
  off += round_up(sizeof(int64_t) * static_cast<size_t>(BT > 0 ? BT : 0), 256);
  w.W = reinterpret_cast<uint16_t*>(p + off);
  (void)H;
  return w;
}

cudaError_t launch_vocab_sort(const FusedArgs& a, const VocabSortWorkspace& w, uint32_t* status, int num_sms,
                              cudaStream_t stream) {
  const int BT = static_cast<int>(a.BT), H = static_cast<int>(a.H), V = static_cast<int>(a.V);
  cudaError_t e;
  hidden_colsum_kernel<<<dim3((H + 255) / 256, kColSplits), 256, 0, stream>>>(a.hidden, BT, H, w.col_part);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  hidden_mean_kernel<<<(H + 255) / 256, 256, 0, stream>>>(w.col_part, BT, H, w.hbar);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int rows_grid = min((V + 7) / 8, num_sms * 8);
  logit_avg_kernel<<<rows_grid, 256, 0, stream>>>(a.W, a.bias, w.hbar, V, H, w.logit_avg, w.keys[0],
                                                         w.vals[0]);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int nb = (V + kSortChunk - 1) / kSortChunk;
  for (int pass = 0; pass < 4; ++pass) {
    const int src = pass & 1;
    radix_hist_kernel<<<nb, kSortThreads, 0, stream>>>(w.keys[src], V, 8 * pass, w.hist);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    radix_scan_kernel<<<1, 256, 0, stream>>>(w.hist, nb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    radix_scatter_kernel<<<nb, kSortThreads, 0, stream>>>(w.keys[src], w.vals[src], V, 8 * pass, w.hist,
                                                          w.keys[src ^ 1], w.vals[src ^ 1]);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // four passes: the sorted order is back in vals[0]
  vocab_gather_kernel<<<rows_grid, 256, 0, stream>>>(a.W, a.bias, w.vals[0], V, H, w.W, w.bias, w.inv, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (BT > 0) {
    target_remap_kernel<<<(BT + 255) / 256, 256, 0, stream>>>(a.target, BT, V, a.ignore_index, w.inv, w.target,
                                                              status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace flce
