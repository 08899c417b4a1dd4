// flce_fwd.cu -- forward passes of fused linear cross-entropy: per-row LSE without logits in HBM.
//
// lse_pair_kernel: one CTA pair (cluster of 2) per (256-token block, vocabulary split).  Each CTA's
// TMA producer warp streams its 128 rows of hidden[k-block] and 128 of the 256 rows of W[n-tile,
// k-block] (128-byte swizzled, 64-wide k-blocks) through a 6-stage mbarrier ring; one thread of the
// even CTA issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16) into one of two 256-column TMEM
// accumulators in each CTA; eight epilogue warps per CTA read each finished tile with tcgen05.ld and
// keep, per row, the online max / sum-exp update ("Fused Linear Cross-Entropy", "Forward -- one
// Triton kernel, online softmax across vocab splits", steps 1-3) and the target logit when the tile
// holds the target column.  Double-buffered accumulators let the epilogue of tile j overlap the MMAs
// of tile j+1.
//
// lse_merge: per row, log-sum-exp merge of the split partials (the partial-LSE combination of "Cut
// Cross Entropy visualized", "Forward kernel", done by ownership instead of a spin lock).
//
// loss_reduce: one CTA sums the per-row loss terms and the valid count in a fixed order.
#include <cstdio>

#include "flce_kernels.cuh"
#include "sm100.cuh"

namespace flce {

namespace {

constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTmemCols = 512;


// Merge of two online (max, sum, weighted sum) states: m in log2 units, s = sum 2^(x - m),
// t = sum 2^(x - m) z (z the logit; used for the entropy).
__device__ __forceinline__ void merge_mst(float& m, float& s, float& t, float m2, float s2, float t2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  const float a = (m == mn) ? 1.f : ex2_approx(m - mn);
  const float b = (m2 == mn) ? 1.f : ex2_approx(m2 - mn);
  m = mn;
  s = s * a + s2 * b;
  t = t * a + t2 * b;
}

// ---------------------------------------------------------------------------------------------------
// lse_pair_kernel: the same pass on CTA pairs (cluster of 2, cta_group::2 MMA, M = 256 tokens per
// pair, N = 256 vocabulary entries per tile).  Each SM streams its own 128 token rows and 128 of the
// tile's 256 vocabulary rows per k-block, half the shared-memory bytes per FLOP of the one-SM tile.
constexpr int kPairStages = 6;
constexpr uint32_t kPairBox = kTileM * kBK * 2;   // 16 KiB
constexpr uint32_t kPairStage = 2 * kPairBox;

struct LsePairSmem {
  uint8_t stage[kPairStages][kPairStage];
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float2 half_ms[kTileM];
  float half_t[kTileM];
};
constexpr size_t kLsePairSmemBytes = sizeof(LsePairSmem) + 1024;
static_assert(kLsePairSmemBytes <= 232448, "shared memory budget of one CTA exceeded");

// kEntropy: also accumulate t = sum 2^(x - m) z per row and split (part_t) for the row entropy.
template <bool kEntropy>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
lse_pair_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
                const float* __restrict__ bias, const int64_t* __restrict__ target, int BT, int V,
                int64_t ignore_index, int num_kb, int tiles_per_split, int n_tiles, int BTp,
                float2* __restrict__ part, float* __restrict__ part_t, float* __restrict__ zy_out,
                uint32_t* __restrict__ status, const uint32_t* __restrict__ gate) {
  // behind an online grad_input pass this launch runs only when that pass asked for it
  if (gate != nullptr && *reinterpret_cast<const volatile uint32_t*>(gate) == 0u) return;
  extern __shared__ uint8_t smem_raw[];
  LsePairSmem& sm =
      *reinterpret_cast<LsePairSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x >> 1) * (2 * kTileM) + static_cast<int>(rank) * kTileM;
  const int split = blockIdx.y;
  const int t_begin = split * tiles_per_split;
  const int nt = max(0, min(n_tiles, t_begin + tiles_per_split) - t_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.acc_full[a], 1);
      mbar_init(&sm.acc_empty[a], 2 * kEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(&sm.tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmap_h);
    tma_prefetch_desc(&tmap_w);
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int j = 0; j < nt && ok; ++j) {
        const int n0 = (t_begin + j) * kBN + static_cast<int>(rank) * kTileM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(smem_u32(&sm.full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2 * kPairStage);
          tma_load_2d_pair(sm.stage[stage], &tmap_h, fb, kb * kBK, r0);
          tma_load_2d_pair(sm.stage[stage] + kPairBox, &tmap_w, fb, kb * kBK, n0);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kTileM, kBN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int j = 0; j < nt && ok; ++j) {
        const int acc = j & 1;
        if (!mbar_wait_cluster(&sm.acc_empty[acc], ((j >> 1) & 1) ^ 1, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sm.stage[stage]);
          const uint32_t b_base = a_base + kPairBox;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ss_pair(d_tmem, sdesc_sw128(a_base + 32u * k, 16u, 1024u),
                             sdesc_sw128(b_base + 32u * k, 16u, 1024u), idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair(&sm.empty[stage]);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit_pair(&sm.acc_full[acc]);
      }
      mma_commit_pair(&sm.drain);
      mbar_wait_drain(&sm.drain, 0);
    }
  } else {
    const int q = warp & 3;
    const int h = warp >> 2;
    const int row_local = q * 32 + lane;
    const int row = r0 + row_local;
    const uint32_t acc_empty_c0 = mapa_shared(smem_u32(&sm.acc_empty[0]), 0);
    const uint32_t acc_empty_c1 = mapa_shared(smem_u32(&sm.acc_empty[1]), 0);
    int64_t y = -1;
    if (row < BT) {
      const int64_t t = target[row];
      if (t != ignore_index && t >= 0 && t < V) y = t;
    }
    const bool has_bias = (bias != nullptr);
    float m = -INFINITY, s = 0.f, t = 0.f, zy = 0.f;
    bool found = false;
    for (int j = 0; j < nt; ++j) {
      const int acc = j & 1;
      if (!mbar_wait(&sm.acc_full[acc], (j >> 1) & 1, abort)) break;
      tc_fence_after();
      const int n0 = (t_begin + j) * kBN + h * 128;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN + h * 128);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(taddr + 32u * c, r);
        tmem_wait_ld();
        const int col0 = n0 + 32 * c;
        // One range test per 32-column chunk: the vocabulary tail and the target column.
        const bool full = col0 + 32 <= V;
        const bool has_y = static_cast<uint64_t>(y - col0) < 32u;
        float x[32];
        float cm = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float v = __uint_as_float(r[i]);
          if (has_bias && (full || col0 + i < V)) v += __ldg(bias + col0 + i);
          if (!full && col0 + i >= V) v = -INFINITY;
          x[i] = v;
          cm = fmaxf(cm, v);
        }
        if (has_y) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col0 + i == static_cast<int>(y)) zy = x[i];
          found = true;
        }
        // log2 e > 0, so the max of the scaled values is the scaled max
        const float mn = fmaxf(m, cm * kLog2e);
        if (mn != -INFINITY) {
          const float resc = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
          float acc_s = s * resc;
          float acc_t = t * resc;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float e = ex2_approx(fmaf(x[i], kLog2e, -mn));
            acc_s += e;
            if (kEntropy) acc_t = fmaf(e, (full || col0 + i < V) ? x[i] : 0.f, acc_t);
          }
          s = acc_s;
          t = acc_t;
          m = mn;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? acc_empty_c1 : acc_empty_c0);
    }
    if (h == 1) {
      sm.half_ms[row_local] = make_float2(m, s);
      if (kEntropy) sm.half_t[row_local] = t;
    }
    named_barrier_sync(1, kEpiWarps * 32);
    if (h == 0) {
      const float2 o = sm.half_ms[row_local];
      merge_mst(m, s, t, o.x, o.y, kEntropy ? sm.half_t[row_local] : 0.f);
      if (row < BT) {
        part[static_cast<size_t>(split) * BTp + row] = make_float2(m, s);
        if (kEntropy) part_t[static_cast<size_t>(split) * BTp + row] = t;
      }
    }
    if (found && row < BT) zy_out[row] = zy;
  }

  tc_fence_before();
  cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) atomicOr(status, kStatusTimeout);
}

// Per row: merge of the split partials into LSE, the row's loss term and the statistics the gradient
// passes read; per vocabulary column: the bias in log2 units, -inf past V.
__global__ void lse_merge_kernel(const float2* __restrict__ part, const float* __restrict__ part_t, int splits, int BTp,
                                 float* __restrict__ entropy, const float* __restrict__ zy,
                                 const int64_t* __restrict__ target, int BT, int V, int64_t ignore_index,
                                 float z_loss, const float* __restrict__ bias, const float* __restrict__ grad_tok,
                                 float4* __restrict__ stats, float2* __restrict__ stats_ct,
                                 float* __restrict__ row_loss, float* __restrict__ loss_tok, float* __restrict__ colb2,
                                 uint32_t* __restrict__ zf_neg, uint32_t* __restrict__ status,
                                 const uint32_t* __restrict__ gate) {
  if (gate != nullptr && *reinterpret_cast<const volatile uint32_t*>(gate) == 0u) return;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  // per-column bias in log2 units for the gradient passes; -inf masks the columns past V
  if (t < ((V + 255) & ~255)) colb2[t] = t < V ? (bias != nullptr ? bias[t] * kLog2e : 0.f) : -INFINITY;
  if (t >= BT) {
    // padding rows (up to a multiple of 256 tokens) read by the gradient passes: no contribution
    if (t < ((BT + 255) & ~255)) {
      stats[t] = make_float4(-INFINITY, __int_as_float(-1), 0.f, 0.f);
      stats_ct[t] = make_float2(-INFINITY, __int_as_float(-1));
    }
    return;
  }
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part[static_cast<size_t>(s) * BTp + t].x);
  float S = 0.f, T = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 p = part[static_cast<size_t>(s) * BTp + t];
    if (p.x != -INFINITY) {
      const float w = exp2f(p.x - M);
      S += p.y * w;
      if (entropy != nullptr) T += part_t[static_cast<size_t>(s) * BTp + t] * w;
    }
  }
  const float lse2 = M + log2f(S);
  const float lse = lse2 * kLn2;
  // entropy of softmax(z_t) = LSE - sum_n p_n z_n, for every row
  if (entropy != nullptr) entropy[t] = lse - T / S;
  const int64_t y = target[t];
  const bool valid = (y != ignore_index) && (y >= 0) && (y < V);
  if (!valid && y != ignore_index) atomicOr(status, kStatusBadTarget);
  const float lt = valid ? (lse - zy[t]) + z_loss * lse * lse : 0.f;
  row_loss[t] = lt;
  if (loss_tok != nullptr) loss_tok[t] = lt;
  // dS of this row = G u f 2^(S log2 e - LSE2) - G u [n = y] with G the scalar gradient scale and u the
  // row's upstream gradient; the log form 2^(S log2 e + log2(u f) - LSE2) needs u f > 0
  const float u = grad_tok != nullptr ? grad_tok[t] : 1.0f;
  const float f = 1.0f + 2.0f * z_loss * lse;
  const float uf = u * f;
  if (valid && u != 0.f && !(uf > 0.f)) atomicOr(zf_neg, 1u);
  const float2 ct = make_float2(valid && uf > 0.f ? log2f(uf) - lse2 : -INFINITY,
                                __int_as_float(valid ? static_cast<int>(y) : -1));
  stats[t] = make_float4(ct.x, ct.y, valid ? u : 0.f, lse2);
  stats_ct[t] = ct;
}

constexpr int kReduceThreads = 1024;

__global__ void __launch_bounds__(kReduceThreads)
loss_reduce_kernel(const float* __restrict__ row_loss, const float4* __restrict__ stats, int BT, int reduction,
                   float grad_scale, float* __restrict__ scale_ws, int64_t* __restrict__ n_valid_ws,
                   uint32_t* __restrict__ zf_neg, float* __restrict__ loss, int64_t* __restrict__ n_valid_out,
                   const uint32_t* __restrict__ gate) {
  if (gate != nullptr && *reinterpret_cast<const volatile uint32_t*>(gate) == 0u) return;
  __shared__ double s_sum[kReduceThreads / 32];
  __shared__ long long s_cnt[kReduceThreads / 32];
  double acc = 0.0;
  long long cnt = 0;
  for (int t = threadIdx.x; t < BT; t += kReduceThreads) {
    acc += static_cast<double>(row_loss[t]);
    cnt += (__float_as_int(stats[t].y) >= 0) ? 1 : 0;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  }
  if ((threadIdx.x & 31) == 0) {
    s_sum[threadIdx.x >> 5] = acc;
    s_cnt[threadIdx.x >> 5] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    long long n = 0;
    for (int w = 0; w < kReduceThreads / 32; ++w) {
      total += s_sum[w];
      n += s_cnt[w];
    }
    const double scale = (reduction == 0) ? 1.0 / static_cast<double>(n > 0 ? n : 1) : 1.0;
    if (loss != nullptr) *loss = static_cast<float>(total * scale);
    // the gradient scale; the log form of dS needs it positive
    const float G = static_cast<float>(scale * static_cast<double>(grad_scale));
    *scale_ws = G;
    if (!(G > 0.f)) *zf_neg |= 1u;
    *n_valid_ws = n;
    if (n_valid_out != nullptr) *n_valid_out = n;
  }
}

// Before an online grad_input pass: the per-column bias table (as lse_merge_kernel writes it) and the
// statistics of the padding rows past BT.
__global__ void online_prep_kernel(const float* __restrict__ bias, int V, int BT, float* __restrict__ colb2,
                                   float4* __restrict__ stats, float2* __restrict__ stats_ct) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < ((V + 255) & ~255)) colb2[t] = t < V ? (bias != nullptr ? bias[t] * kLog2e : 0.f) : -INFINITY;
  if (t >= BT && t < ((BT + 255) & ~255)) {
    stats[t] = make_float4(-INFINITY, __int_as_float(-1), 0.f, 0.f);
    stats_ct[t] = make_float2(-INFINITY, __int_as_float(-1));
  }
}

// Before an online grad_input pass (one CTA): the valid count, the gradient scale G and the bad-target
// flag, from the targets alone (the loss reduction after the pass computes the same count and G again).
__global__ void __launch_bounds__(kReduceThreads)
online_count_kernel(const int64_t* __restrict__ target, int BT, int V, int64_t ignore_index, int reduction,
                    float grad_scale, float* __restrict__ scale_ws, uint32_t* __restrict__ zf_neg,
                    uint32_t* __restrict__ status) {
  __shared__ long long s_cnt[kReduceThreads / 32];
  long long cnt = 0;
  bool bad = false;
  for (int t = threadIdx.x; t < BT; t += kReduceThreads) {
    const int64_t y = target[t];
    const bool valid = (y != ignore_index) && (y >= 0) && (y < V);
    cnt += valid ? 1 : 0;
    bad |= !valid && y != ignore_index;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusBadTarget);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long n = 0;
    for (int w = 0; w < kReduceThreads / 32; ++w) n += s_cnt[w];
    const double scale = (reduction == 0) ? 1.0 / static_cast<double>(n > 0 ? n : 1) : 1.0;
    const float G = static_cast<float>(scale * static_cast<double>(grad_scale));
    *scale_ws = G;
    if (!(G > 0.f)) *zf_neg |= 1u;
  }
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int choose_splits(int m_tiles, int n_tiles, int num_sms) {
  // Pick the split count whose grid fills the SMs best (waves rounded up), preferring fewer splits.
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= kMaxSplits && s <= n_tiles; ++s) {
    const int tps = (n_tiles + s - 1) / s;
    const int real = (n_tiles + tps - 1) / tps;
    const long long ctas = static_cast<long long>(m_tiles) * real;
    const long long waves = (ctas + num_sms - 1) / num_sms;
    // work per CTA is tps tiles; the busiest SM does waves * tps tiles; ideal is m_tiles*n_tiles/num_sms
    const double ideal = static_cast<double>(m_tiles) * n_tiles / num_sms;
    const double eff = ideal / static_cast<double>(waves * tps);
    if (eff > best_eff + 1e-3) {
      best_eff = eff;
      best = real;
    }
  }
  return best;
}

}  // namespace

size_t fused_workspace_bytes(int64_t BT, int64_t V) {
  const size_t btp = align_up(static_cast<size_t>(BT > 0 ? BT : 0), kTileM);
  const size_t vp = align_up(static_cast<size_t>(V > 0 ? V : 0), 256);
  size_t off = 256;
  off += align_up(sizeof(float2) * kMaxSplits * btp, 256);
  off += align_up(sizeof(float) * kMaxSplits * btp, 256);
  off += align_up(sizeof(float) * btp, 256);
  off += align_up(sizeof(float4) * align_up(btp, 256), 256);
  off += align_up(sizeof(float2) * align_up(btp, 256), 256);
  off += align_up(sizeof(float) * btp, 256);
  off += align_up(sizeof(float) * vp, 256);
  off += align_up(sizeof(uint32_t) * btp, 256);
  off += sizeof(float) * kMaxSplitUnits * 256;
  off += sizeof(float4) * kMaxSplitUnits * 256 * 8;
  off += sizeof(float4) * kMaxSplitUnits * 256;
  off += kSplitAccBytes;
  return off;
}

FusedWorkspace carve_workspace(void* base, int64_t BT, int64_t V) {
  const size_t vp = align_up(static_cast<size_t>(V > 0 ? V : 0), 256);
  const size_t btp = align_up(static_cast<size_t>(BT > 0 ? BT : 0), kTileM);
  auto* p = static_cast<unsigned char*>(base);
  FusedWorkspace w;
  w.status = reinterpret_cast<uint32_t*>(p);
  w.scale = reinterpret_cast<float*>(p + 4);
  w.n_valid = reinterpret_cast<int64_t*>(p + 8);
  w.zf_neg = reinterpret_cast<uint32_t*>(p + 16);
  w.skipped = reinterpret_cast<uint32_t*>(p + 20);
  w.fallback = reinterpret_cast<uint32_t*>(p + 24);
  w.vs_count = reinterpret_cast<uint32_t*>(p + 28);
  w.ts_count = reinterpret_cast<uint32_t*>(p + 32);
  w.work_q = reinterpret_cast<unsigned long long*>(p + 40);
  w.side_count = reinterpret_cast<uint32_t*>(p + 56);
  w.single_units = reinterpret_cast<uint32_t*>(p + 64);
  w.single_count = reinterpret_cast<uint32_t*>(p + 72);
  size_t off = 256;
  w.part = reinterpret_cast<float2*>(p + off);
  w.part_bytes = align_up(sizeof(float2) * kMaxSplits * btp, 256);
  off += w.part_bytes;
  w.part_t = reinterpret_cast<float*>(p + off);
  off += align_up(sizeof(float) * kMaxSplits * btp, 256);
  w.zy = reinterpret_cast<float*>(p + off);
  off += align_up(sizeof(float) * btp, 256);
  w.stats = reinterpret_cast<float4*>(p + off);
  off += align_up(sizeof(float4) * align_up(btp, 256), 256);
  w.stats_ct = reinterpret_cast<float2*>(p + off);
  off += align_up(sizeof(float2) * align_up(btp, 256), 256);
  w.row_loss = reinterpret_cast<float*>(p + off);
  off += align_up(sizeof(float) * btp, 256);
  w.colb2 = reinterpret_cast<float*>(p + off);
  off += align_up(sizeof(float) * vp, 256);
  w.row_redo = reinterpret_cast<uint32_t*>(p + off);
  off += align_up(sizeof(uint32_t) * btp, 256);
  w.vs_mref = reinterpret_cast<float*>(p + off);
  off += sizeof(float) * kMaxSplitUnits * 256;
  w.vs_part = reinterpret_cast<float4*>(p + off);
  off += sizeof(float4) * kMaxSplitUnits * 256 * 8;
  w.vs_stat = reinterpret_cast<float4*>(p + off);
  off += sizeof(float4) * kMaxSplitUnits * 256;
  w.split_acc = reinterpret_cast<float*>(p + off);
  return w;
}

cudaError_t launch_lse_passes(const FusedArgs& a, const FusedWorkspace& ws, int num_sms, cudaStream_t stream,
                              char* err, size_t err_len, cudaEvent_t const* events, const uint32_t* gate) {
  const int BT = static_cast<int>(a.BT);
  const int V = static_cast<int>(a.V);
  const int BTp = static_cast<int>(align_up(static_cast<size_t>(BT), kTileM));
  cudaError_t e;
  if (BT > 0) {
    CUtensorMap tm_h, tm_w;
    if (!make_tmap_bf16(&tm_h, a.hidden, a.BT, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tm_w, a.W, a.V, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
    const int pairs = (BT + 2 * kTileM - 1) / (2 * kTileM);
    const int n_tiles = (V + kBN - 1) / kBN;
    const int splits = choose_splits(pairs, n_tiles, num_sms / 2);
    const int tps = (n_tiles + splits - 1) / splits;
    const int num_kb = static_cast<int>((a.H + kBK - 1) / kBK);
    const bool want_entropy = (a.entropy != nullptr);
    auto kern = want_entropy ? lse_pair_kernel<true> : lse_pair_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kLsePairSmemBytes));
    if (e != cudaSuccess) return e;
    kern<<<dim3(2 * pairs, splits), kThreads, kLsePairSmemBytes, stream>>>(
        tm_h, tm_w, a.bias, a.target, BT, V, a.ignore_index, num_kb, tps, n_tiles, BTp, ws.part, ws.part_t, ws.zy,
        ws.status, gate);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (events != nullptr && (e = cudaEventRecord(events[1], stream)) != cudaSuccess) return e;
    const int merge_threads = max((BT + 255) & ~255, (V + 255) & ~255);
    lse_merge_kernel<<<merge_threads / 256, 256, 0, stream>>>(ws.part, ws.part_t, splits, BTp, a.entropy, ws.zy,
                                                            a.target, BT, V,
                                                            a.ignore_index, a.z_loss, a.bias, a.grad_tok, ws.stats,
                                                            ws.stats_ct, ws.row_loss, a.loss_tok, ws.colb2, ws.zf_neg, ws.status,
                                                            gate);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else if (events != nullptr && (e = cudaEventRecord(events[1], stream)) != cudaSuccess) {
    return e;
  }
  loss_reduce_kernel<<<1, kReduceThreads, 0, stream>>>(ws.row_loss, ws.stats, BT, a.reduction, a.grad_scale, ws.scale,
                                                      ws.n_valid, ws.zf_neg, a.loss, a.n_valid_out, gate);
  return cudaGetLastError();
}

cudaError_t launch_online_prep(const FusedArgs& a, const FusedWorkspace& ws, cudaStream_t stream) {
  const int BT = static_cast<int>(a.BT);
  const int V = static_cast<int>(a.V);
  const int n = max((BT + 255) & ~255, (V + 255) & ~255);
  online_prep_kernel<<<n / 256, 256, 0, stream>>>(a.bias, V, BT, ws.colb2, ws.stats, ws.stats_ct);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  online_count_kernel<<<1, kReduceThreads, 0, stream>>>(a.target, BT, V, a.ignore_index, a.reduction, a.grad_scale,
                                                       ws.scale, ws.zf_neg, ws.status);
  return cudaGetLastError();
}

cudaError_t launch_loss_reduce(const FusedArgs& a, const FusedWorkspace& ws, cudaStream_t stream) {
  loss_reduce_kernel<<<1, kReduceThreads, 0, stream>>>(ws.row_loss, ws.stats, static_cast<int>(a.BT), a.reduction,
                                                      a.grad_scale, ws.scale, ws.n_valid, ws.zf_neg, a.loss,
                                                      a.n_valid_out, nullptr);
  return cudaGetLastError();
}

}  // namespace flce
