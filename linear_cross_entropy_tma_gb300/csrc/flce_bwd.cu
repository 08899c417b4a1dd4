// flce_bwd.cu -- backward passes of fused linear cross-entropy with dlogits kept on chip.
//
// Both gradients have the shape of one "attention-like" loop in which the operand that produces the
// logits tile is also the operand the gradient GEMM consumes:
//
//   grad_input[m, :] = sum_n dS[m, n] W[n, :]         rows = tokens,     columns = vocabulary
//   grad_W[n, :]     = sum_m dS[m, n]^T hidden[m, :]  rows = vocabulary, columns = tokens
//
// with dS[m, n] = s [y_m valid] (exp(z[m, n] - LSE_m) (1 + 2 z_loss LSE_m) - [n = y_m])
// ("Fused Linear Cross-Entropy", "From dlogits to grad_input and grad_W"; the recompute-with-saved-
// statistics scheme of "Why two passes ..." option 2 and of "Cut Cross Entropy visualized",
// "Backward pass", steps 2-6).
//
// One CTA owns a 128-row tile of the output and a chunk of up to 256 of its H columns, and walks the
// whole reduction dimension in 128-wide column tiles:
//   GEMM1  S = rows[128, H] . cols[128, H]^T          -> TMEM (two 128-column buffers)
//   epi    dS = f(S, per-row / per-column statistics)  -> registers -> bf16 in shared memory
//          (128-byte-swizzled K-major layout, the A operand of the next MMA; never written to HBM)
//   GEMM2  O[128, Hc] += dS[128, 128] . cols[128, Hc]  -> TMEM (Hc <= 256 columns, fp32)
// The cols operand of GEMM2 is the same matrix as GEMM1's B operand, read MN-major.  The pipeline
// runs GEMM1 of tile j+1 while the epilogue turns tile j into dS, then GEMM2 of tile j.  At the end
// the fp32 accumulator is written out once: bf16 grad_input, or fp32 grad_W plus grad_bias (the
// row sums of dS in fp32).
//
// H wider than 256 is covered by several CTAs per row tile, each recomputing the logits tile for
// its own H chunk.
#include "flce_kernels.cuh"
#include "sm100.cuh"

namespace flce {

cudaError_t launch_lse_passes(const FusedArgs& a, const FusedWorkspace& ws, int num_sms, cudaStream_t stream,
                              char* err, size_t err_len, cudaEvent_t const* events);

namespace {

constexpr int kBN = 128;              // logits tile columns = K extent of GEMM2 per tile
constexpr int kBK = 64;
constexpr int kHc = 256;              // H columns per CTA (GEMM2 N)
constexpr int kStages = 4;
constexpr uint32_t kHalf = kTileM * kBK * 2;   // 16 KiB: one 128 x 64 bf16 box
constexpr uint32_t kStageBytes = 2 * kHalf;    // GEMM1: A + B; GEMM2: up to 4 boxes of 64 x 64
constexpr uint32_t kBox2 = 64 * 64 * 2;        // 8 KiB
constexpr uint32_t kDsBytes = kTileM * kBN * 2;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 2 * kBN;           // O accumulator starts after the two S buffers

struct DgSmem {
  uint8_t stage[kStages][kStageBytes];
  uint8_t ds[2][kDsBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t ds_full[2];
  uint64_t ds_empty[2];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float half_bias[kTileM];
};
constexpr size_t kDgSmemBytes = sizeof(DgSmem) + 1024;

struct DgParams {
  const float* bias;
  const float4* stats;      // per token: (LSE log2e, 1 + 2 z_loss LSE, valid, target bits)
  const float* scale;       // s
  int BT, V, H;
  int n_rows;               // rows of the output (BT for grad_input, V for grad_W)
  int n_cols;               // reduction length (V for grad_input, BT for grad_W)
  int num_kb;               // ceil(H / 64)
  uint16_t* grad_input;     // rows = tokens
  float* grad_W;            // rows = vocabulary
  float* grad_bias;
};

// kVocabRows = false: rows are tokens (grad_input pass); true: rows are vocabulary entries (grad_W).
template <bool kVocabRows>
__global__ void __launch_bounds__(kThreads, 1)
dgrad_kernel(const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_cols,
             const __grid_constant__ CUtensorMap tm_cols64, const DgParams p, uint32_t* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  DgSmem& sm = *reinterpret_cast<DgSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kTileM;           // first output row of this CTA
  const int h0 = blockIdx.y * kHc;              // first H column of this CTA
  const int hc = min(kHc, p.H - h0);            // H columns owned (multiple of 8)
  const int n_box = (hc + 63) / 64;             // 64-wide boxes of the GEMM2 B operand
  const uint32_t n2 = static_cast<uint32_t>((hc + 15) / 16 * 16);
  const int nt = (p.n_cols + kBN - 1) / kBN;    // column tiles along the reduction

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.s_empty[b], kEpiWarps);
      mbar_init(&sm.ds_full[b], kEpiWarps);
      mbar_init(&sm.ds_empty[b], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_rows);
    tma_prefetch_desc(&tm_cols);
    tma_prefetch_desc(&tm_cols64);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_phase = 0;
      bool ok = true;
      auto next = [&]() {
        filled |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      };
      auto load_gemm1 = [&](int j) {
        for (int kb = 0; kb < p.num_kb && ok; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
            ok = false;
            return;
          }
          mbar_arrive_expect_tx(&sm.full[stage], kStageBytes);
          tma_load_2d(sm.stage[stage], &tm_rows, &sm.full[stage], kb * kBK, r0);
          tma_load_2d(sm.stage[stage] + kHalf, &tm_cols, &sm.full[stage], kb * kBK, j * kBN);
          next();
        }
      };
      auto load_gemm2 = [&](int j) {
        for (int half = 0; half < 2 && ok; ++half) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
            ok = false;
            return;
          }
          mbar_arrive_expect_tx(&sm.full[stage], static_cast<uint32_t>(n_box) * kBox2);
          for (int b = 0; b < n_box; ++b)
            tma_load_2d(sm.stage[stage] + b * kBox2, &tm_cols64, &sm.full[stage], h0 + 64 * b, j * kBN + 64 * half);
          next();
        }
      };
      for (int j = 0; j < nt && ok; ++j) {
        load_gemm1(j);
        if (j >= 1) load_gemm2(j - 1);
      }
      if (ok) load_gemm2(nt - 1);
      if (!ok) {
        for (int s = 0; s < kStages; ++s)
          if (filled & (1u << s)) mbar_wait_drain(&sm.full[s], (last_phase >> s) & 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc1 = idesc_bf16_f32(kTileM, kBN, false, false);
      const uint32_t idesc2 = idesc_bf16_f32(kTileM, n2, false, true);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      auto advance = [&]() {
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      };
      auto gemm2 = [&](int i) {
        const int b = i & 1;
        if (!mbar_wait(&sm.ds_full[b], (i >> 1) & 1, abort)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sm.ds[b]);
        for (int half = 0; half < 2; ++half) {
          if (!mbar_wait(&sm.full[stage], phase, abort)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t b_base = smem_u32(sm.stage[stage]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = sdesc_sw128(a_base + half * kHalf + 32u * k, 16u, 1024u);
            const uint64_t bd = sdesc_sw128(b_base + 2048u * k, kBox2, 1024u);
            mma_bf16_ss(tmem + kTmemO, ad, bd, idesc2, (i | half | k) != 0 ? 1u : 0u);
          }
          mma_commit(&sm.empty[stage]);
          advance();
        }
        mma_commit(&sm.ds_empty[b]);
      };
      for (int j = 0; j < nt && ok; ++j) {
        const int acc = j & 1;
        if (!mbar_wait(&sm.s_empty[acc], ((j >> 1) & 1) ^ 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sm.stage[stage]);
          const uint32_t b_base = a_base + kHalf;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ss(d_tmem, sdesc_sw128(a_base + 32u * k, 16u, 1024u), sdesc_sw128(b_base + 32u * k, 16u, 1024u),
                        idesc1, (kb | k) != 0 ? 1u : 0u);
          mma_commit(&sm.empty[stage]);
          advance();
        }
        if (!ok) break;
        mma_commit(&sm.s_full[acc]);
        if (j >= 1) gemm2(j - 1);
      }
      if (ok) gemm2(nt - 1);
      if (ok) mma_commit(&sm.o_full);
      mma_commit(&sm.drain);
      mbar_wait_drain(&sm.drain, 0);
    }
  } else {
    // ---------------------------------------------------------------------------- epilogue warps
    const int q = warp & 3;
    const int hh = warp >> 2;                  // which 64-column half of the 128-wide tile
    const int rl = q * 32 + lane;              // row within the tile = TMEM lane
    const int row = r0 + rl;
    const float scale = *p.scale;
    // per-row constants
    float row_lse2 = 0.f, row_zf = 0.f, row_coef = 0.f, row_bias2 = 0.f;
    int row_y = -1;
    if (!kVocabRows) {
      if (row < p.BT) {
        const float4 st = p.stats[row];
        row_lse2 = st.x;
        row_zf = st.y;
        row_coef = st.z * scale;
        row_y = __float_as_int(st.w);
      }
    } else {
      if (p.bias != nullptr && row < p.V) row_bias2 = __ldg(p.bias + row) * kLog2e;
    }
    float gbias = 0.f;
    bool ok = true;
    uint8_t* const ds_row_base0 = sm.ds[0] + hh * kHalf + rl * 128;
    uint8_t* const ds_row_base1 = sm.ds[1] + hh * kHalf + rl * 128;
    for (int j = 0; j < nt; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&sm.s_full[b], (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[64];
      {
        const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * kBN + hh * 64);
        uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
        uint32_t (&rb)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
        tmem_ld_32cols(taddr, ra);
        tmem_ld_32cols(taddr + 32u, rb);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_empty[b]);

      const int col0 = j * kBN + hh * 64;
      uint32_t packed[32];
#pragma unroll
      for (int i2 = 0; i2 < 32; ++i2) {
        float d[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = 2 * i2 + u;
          const int col = col0 + i;
          const float sv = __uint_as_float(r[i]);
          float g;
          if (!kVocabRows) {
            // rows = tokens, columns = vocabulary entries
            const float b2 = (p.bias != nullptr && col < p.V) ? __ldg(p.bias + col) * kLog2e : 0.f;
            const float e = ex2_approx(fmaf(sv, kLog2e, b2 - row_lse2)) * row_zf;
            g = row_coef * (col == row_y ? e - 1.0f : e);
          } else {
            // rows = vocabulary entries, columns = tokens
            float4 st = make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
            if (col < p.BT) st = __ldg(p.stats + col);
            const float e = ex2_approx(fmaf(sv, kLog2e, row_bias2 - st.x)) * st.y;
            g = (st.z * scale) * (__float_as_int(st.w) == row ? e - 1.0f : e);
            gbias += g;
          }
          d[u] = g;
        }
        packed[i2] = pack_bf16x2(d[0], d[1]);
      }
      // the GEMM2 that read this dS buffer two tiles ago must be done
      if (!mbar_wait(&sm.ds_empty[b], ((j >> 1) & 1) ^ 1, abort)) {
        ok = false;
        break;
      }
      uint8_t* dst = b ? ds_row_base1 : ds_row_base0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        *reinterpret_cast<uint4*>(dst + ((c ^ (rl & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.ds_full[b]);
    }

    if (ok && mbar_wait(&sm.o_full, 0, abort)) {
      tc_fence_after();
      const int n_chunks = (hc + 31) / 32;
      for (int c = hh; c < n_chunks; c += 2) {
        uint32_t v[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(q * 32) << 16) + kTmemO + 32u * c, v);
        tmem_wait_ld();
        const int cb = 32 * c;  // column within the chunk of H
        if (!kVocabRows) {
          if (row < p.BT) {
            uint16_t* out = p.grad_input + static_cast<size_t>(row) * p.H + h0 + cb;
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              if (cb + 8 * g8 + 8 <= hc) {
                const uint4 w = make_uint4(pack_bf16x2(__uint_as_float(v[8 * g8 + 0]), __uint_as_float(v[8 * g8 + 1])),
                                           pack_bf16x2(__uint_as_float(v[8 * g8 + 2]), __uint_as_float(v[8 * g8 + 3])),
                                           pack_bf16x2(__uint_as_float(v[8 * g8 + 4]), __uint_as_float(v[8 * g8 + 5])),
                                           pack_bf16x2(__uint_as_float(v[8 * g8 + 6]), __uint_as_float(v[8 * g8 + 7])));
                *reinterpret_cast<uint4*>(out + 8 * g8) = w;
              }
            }
          }
        } else {
          if (row < p.V && p.grad_W != nullptr) {
            float* out = p.grad_W + static_cast<size_t>(row) * p.H + h0 + cb;
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
              if (cb + 4 * g4 + 4 <= hc) {
                *reinterpret_cast<float4*>(out + 4 * g4) =
                    make_float4(__uint_as_float(v[4 * g4 + 0]), __uint_as_float(v[4 * g4 + 1]),
                                __uint_as_float(v[4 * g4 + 2]), __uint_as_float(v[4 * g4 + 3]));
              }
            }
          }
        }
      }
    }
    if (kVocabRows) {
      if (hh == 1) sm.half_bias[rl] = gbias;
      named_barrier_sync(1, kEpiWarps * 32);
      if (hh == 0 && ok && blockIdx.y == 0 && p.grad_bias != nullptr && row < p.V)
        p.grad_bias[row] = gbias + sm.half_bias[rl];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) atomicOr(status, kStatusTimeout);
}

template <bool kVocabRows>
cudaError_t launch_dgrad(const CUtensorMap& rows, const CUtensorMap& cols, const CUtensorMap& cols64,
                         const DgParams& p, uint32_t* status, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(dgrad_kernel<kVocabRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDgSmemBytes));
  if (e != cudaSuccess) return e;
  // with only grad_bias requested one H chunk suffices (the GEMM2 result is not stored)
  const int h_chunks = (kVocabRows && p.grad_W == nullptr) ? 1 : (p.H + kHc - 1) / kHc;
  const dim3 grid((p.n_rows + kTileM - 1) / kTileM, h_chunks);
  dgrad_kernel<kVocabRows><<<grid, kThreads, kDgSmemBytes, stream>>>(rows, cols, cols64, p, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, void* workspace, int num_sms, cudaStream_t stream, char* err,
                         size_t err_len, cudaEvent_t const* events) {
  const FusedWorkspace ws = carve_workspace(workspace, a.BT);
  auto mark = [&](int i) { return events != nullptr ? cudaEventRecord(events[i], stream) : cudaSuccess; };
  cudaError_t e = cudaMemsetAsync(workspace, 0, 256, stream);
  if (e != cudaSuccess) return e;
  if ((e = mark(0)) != cudaSuccess) return e;
  if ((e = launch_lse_passes(a, ws, num_sms, stream, err, err_len, events)) != cudaSuccess) return e;
  if ((e = mark(2)) != cudaSuccess) return e;

  const bool want_dw = (a.grad_W != nullptr) || (a.grad_bias != nullptr);
  if (a.BT == 0) {
    // no tokens: every gradient is zero
    if (a.grad_W != nullptr && (e = cudaMemsetAsync(a.grad_W, 0, sizeof(float) * a.V * a.H, stream)) != cudaSuccess)
      return e;
    if (a.grad_bias != nullptr && (e = cudaMemsetAsync(a.grad_bias, 0, sizeof(float) * a.V, stream)) != cudaSuccess)
      return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    return mark(4);
  }
  DgParams p{};
  p.bias = a.bias;
  p.stats = ws.stats;
  p.scale = ws.scale;
  p.BT = static_cast<int>(a.BT);
  p.V = static_cast<int>(a.V);
  p.H = static_cast<int>(a.H);
  p.num_kb = static_cast<int>((a.H + kBK - 1) / kBK);
  p.grad_input = a.grad_input;
  p.grad_W = a.grad_W;
  p.grad_bias = a.grad_bias;
  CUtensorMap tm_h128, tm_w128, tm_h64, tm_w64;
  if (a.grad_input != nullptr || want_dw) {
    if (!make_tmap_bf16(&tm_h128, a.hidden, a.BT, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tm_w128, a.W, a.V, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
  }
  if (a.grad_input != nullptr) {
    if (!make_tmap_bf16(&tm_w64, a.W, a.V, a.H, 64, err, err_len)) return cudaErrorInvalidValue;
    p.n_rows = p.BT;
    p.n_cols = p.V;
    if ((e = launch_dgrad<false>(tm_h128, tm_w128, tm_w64, p, ws.status, stream)) != cudaSuccess) return e;
  }
  if ((e = mark(3)) != cudaSuccess) return e;
  if (want_dw) {
    if (!make_tmap_bf16(&tm_h64, a.hidden, a.BT, a.H, 64, err, err_len)) return cudaErrorInvalidValue;
    p.n_rows = p.V;
    p.n_cols = p.BT;
    if ((e = launch_dgrad<true>(tm_w128, tm_h128, tm_h64, p, ws.status, stream)) != cudaSuccess) return e;
  }
  return mark(4);
}

}  // namespace flce
