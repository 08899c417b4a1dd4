// flce_bwd.cu -- the gradient passes of fused linear cross-entropy on clusters of CTA pairs.
//
// Computation ("Fused Linear Cross-Entropy", "From dlogits to grad_input and grad_W"; logits recompute
// with saved row statistics as in "Cut Cross Entropy visualized", "Backward pass"):
//
//   grad_input[m, :] = sum_n dS[m, n] W[n, :]          rows = tokens,     columns = vocabulary
//   grad_W[n, :]     = sum_m dS[m, n] hidden[m, :]     rows = vocabulary, columns = tokens
//   dS[m, n] = s [y_m valid] (exp(z[m, n] - LSE_m) (1 + 2 z_loss LSE_m) - [n = y_m])
//
// Mapping onto GB300:
//   * A CTA pair (cluster ranks 2p, 2p+1) owns 256 output rows (128 per CTA) and one 256-wide chunk of
//     H.  Its MMAs are cta_group::2: issued by the even CTA, A rows from each CTA's own shared memory,
//     B split by N across the two CTAs, each CTA's 128 result rows in its own tensor memory.
//   * A cluster holds P pairs with the same 256 rows and P different H chunks.  The logits tile of
//     column block j is computed once, by pair (j mod P):
//       GEMM1   S[256, 256] = rows[256, H] . cols[256, H]^T          (TMEM, 256 columns)
//       epi     dS = f(S, statistics) in registers -> bf16 in shared memory, in the 128-byte-swizzled
//               K-major layout of the next MMA's A operand; then copied with cp.async.bulk into the
//               same buffer of the other P-1 pairs' CTAs (distributed shared memory, never HBM)
//     and every pair accumulates its own H chunk:
//       GEMM2   O[256, 256] += dS[256, 256] . cols[256, chunk]      (TMEM, 256 columns, fp32)
//     So the logits of each (row block, column block) are computed ceil(H / (256 P)) times instead of
//     ceil(H / 256) times.
//   * dS buffers form a ring of one or two per CTA: every pair's GEMM2 of block j commits, with
//     multicast to all CTAs of the cluster, on that buffer's "ds_free"; the owner of the next block
//     that uses the buffer writes and sends only after all P commits.
//   * grad_bias (vocabulary rows) is each CTA's fp32 row sum of dS over the blocks it owns, gathered
//     across the pairs in distributed shared memory and added in pair order (deterministic).
// All waits are bounded; a wait that gives up flags the status word and the kernel winds down.
#include "flce_kernels.cuh"
#include "sm100.cuh"

namespace flce {

namespace {

constexpr int kPN = 256;                      // logits tile columns = K of GEMM2 per block
constexpr int kBK = 64;
constexpr int kHc = 256;                      // H columns per pair (GEMM2 N)
// Pairs per cluster.  Sharing logits tiles across P > 1 pairs is implemented and correct, but on GB300
// it measured slower than recomputing them (P = 2: 68 ms vs 62 ms clock-adjusted per gradient pass at
// the long workload; P = 4: 106 ms): a pair's in-order MMA stream can hold the GEMM2 another pair is
// waiting for behind an 8192-cycle GEMM1, and the distributed-shared-memory copies run near 25 B/clk
// per SM.  One pair per cluster is used.
constexpr int kMaxPairs = 1;
constexpr uint32_t kBox = kTileM * kBK * 2;   // 16 KiB: a 128-row x 64-column bf16 box
constexpr uint32_t kStage = 2 * kBox;
constexpr uint32_t kDsBytes = kTileM * kPN * 2;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;

// Shared memory per CTA: an operand ring (5 stages of 32 KiB for the grad_input pass, 4 for the grad_W
// pass, which also stages each owned block's 256 per-token statistics in a two-slot ring and gathers
// grad_bias partials) and the dS buffer ring (kDsBuf buffers of 64 KiB; two allow block j+1 to be
// produced and sent while the pairs' GEMM2 still read block j, measured no faster at P = 1).
template <bool kVocabRows>
struct PairCfg {
  static constexpr int kDsBuf = 1;                         // dS buffers (a ring) per CTA
  static constexpr int kStages = kVocabRows ? 4 : 5;
  static constexpr int kStatSlots = kVocabRows ? 2 : 1;
  static constexpr int kStatCols = kVocabRows ? kPN : 4;
  static constexpr int kGather = kVocabRows ? kMaxPairs : 1;
};

template <bool kVocabRows>
struct PairSmem {
  uint8_t stage[PairCfg<kVocabRows>::kStages][kStage];
  uint8_t ds[PairCfg<kVocabRows>::kDsBuf][kDsBytes];
  float4 colstats[PairCfg<kVocabRows>::kStatSlots][PairCfg<kVocabRows>::kStatCols];
  float gb_gather[PairCfg<kVocabRows>::kGather][kTileM];
  uint64_t full[PairCfg<kVocabRows>::kStages];
  uint64_t empty[PairCfg<kVocabRows>::kStages];
  uint64_t st_full[2];
  uint64_t st_empty[2];
  uint64_t s_full;
  uint64_t s_empty;
  uint64_t ds_full[PairCfg<kVocabRows>::kDsBuf];
  uint64_t ds_free[PairCfg<kVocabRows>::kDsBuf];
  uint64_t rx_full[PairCfg<kVocabRows>::kDsBuf];
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float half_bias[kTileM];
};
template <bool kVocabRows>
constexpr size_t pair_smem_bytes() { return sizeof(PairSmem<kVocabRows>) + 1024; }
static_assert(pair_smem_bytes<false>() <= 232448, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<true>() <= 232448, "shared memory budget of one CTA exceeded");

struct PairParams {
  const float* bias;
  const float4* stats;
  const float* scale;
  int BT, V, H;
  int n_rows, n_cols, num_kb;
  int P;                    // pairs per cluster
  uint16_t* grad_input;
  float* grad_W;
  float* grad_bias;
};

template <bool kVocabRows>
__global__ void __launch_bounds__(kThreads, 1)
dgrad_pair_kernel(const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_cols,
                  const PairParams p, uint32_t* __restrict__ status) {
  constexpr int kStages = PairCfg<kVocabRows>::kStages;
  constexpr int kDsBuf = PairCfg<kVocabRows>::kDsBuf;
  extern __shared__ uint8_t smem_raw[];
  PairSmem<kVocabRows>& sm =
      *reinterpret_cast<PairSmem<kVocabRows>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t rank = cluster_ctarank();
  const int P = p.P;
  const int pr = static_cast<int>(rank >> 1);       // pair index within the cluster
  const uint32_t q = rank & 1u;                     // half of the pair (which 128 rows)
  const bool leader = (q == 0);
  const uint32_t lead_rank = rank & ~1u;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << (2 * pr));
  const uint16_t all_mask = static_cast<uint16_t>((1u << (2 * P)) - 1u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x / (2 * P)) * (2 * kTileM) + static_cast<int>(q) * kTileM;
  const int h0 = (blockIdx.y * P + pr) * kHc;
  const int hc = min(kHc, p.H - h0);
  const uint32_t n2 = hc > 128 ? 256u : 128u;   // GEMM2 N; columns past H are zero-filled by TMA
  const int nbox2 = static_cast<int>(n2) / 128; // 64-column boxes per CTA per GEMM2 stage
  const int nt = (p.n_cols + kPN - 1) / kPN;
  auto owned = [&](int j) { return (j % P) == pr; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.st_full[b], 1);
      mbar_init(&sm.st_empty[b], kEpiWarps);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_empty, 2 * kEpiWarps);
    for (int b = 0; b < kDsBuf; ++b) {
      mbar_init(&sm.ds_full[b], 2);
      mbar_init(&sm.ds_free[b], static_cast<uint32_t>(P));
      mbar_init(&sm.rx_full[b], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(&sm.tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_rows);
    tma_prefetch_desc(&tm_cols);
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
      auto next = [&]() {
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      };
      auto load_gemm1 = [&](int j, int u) {
        if (kVocabRows) {
          // this block's per-token statistics (stats is padded to a multiple of 256 tokens)
          const int sb = u & 1;
          if (!mbar_wait(&sm.st_empty[sb], ((u >> 1) & 1) ^ 1, abort)) {
            ok = false;
            return;
          }
          mbar_arrive_expect_tx(&sm.st_full[sb], kPN * sizeof(float4));
          bulk_load_1d(sm.colstats[sb], p.stats + static_cast<size_t>(j) * kPN, kPN * sizeof(float4), &sm.st_full[sb]);
        }
        for (int kb = 0; kb < p.num_kb && ok; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
            ok = false;
            return;
          }
          const uint32_t fb = mapa_shared(smem_u32(&sm.full[stage]), lead_rank);
          if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2 * kStage);
          tma_load_2d_pair(sm.stage[stage], &tm_rows, fb, kb * kBK, r0);
          tma_load_2d_pair(sm.stage[stage] + kBox, &tm_cols, fb, kb * kBK, j * kPN + static_cast<int>(q) * kTileM);
          next();
        }
      };
      auto load_gemm2 = [&](int j) {
        for (int half = 0; half < 2 && ok; ++half) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
            ok = false;
            return;
          }
          const uint32_t fb = mapa_shared(smem_u32(&sm.full[stage]), lead_rank);
          if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2u * nbox2 * kBox);
          for (int b = 0; b < nbox2; ++b)
            tma_load_2d_pair(sm.stage[stage] + b * kBox, &tm_cols, fb,
                             h0 + static_cast<int>(q * (n2 / 2)) + 64 * b, j * kPN + half * kTileM);
          next();
        }
      };
      int u = 0;
      for (int j = 0; j < nt && ok; ++j) {
        if (owned(j)) load_gemm1(j, u++);
        if (j >= 1) load_gemm2(j - 1);
      }
      if (ok) load_gemm2(nt - 1);
      if (!ok) {
        // let copies already issued land before the CTA can finish
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc1 = idesc_bf16_f32(2 * kTileM, kPN, false, false);
      const uint32_t idesc2 = idesc_bf16_f32(2 * kTileM, n2, false, true);
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
        const int db = i % kDsBuf;
        if (!mbar_wait_cluster(&sm.ds_full[db], (i / kDsBuf) & 1, abort)) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(sm.ds[db]);
        for (int half = 0; half < 2; ++half) {
          if (!mbar_wait(&sm.full[stage], phase, abort)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t b_base = smem_u32(sm.stage[stage]);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = sdesc_sw128(a_base + (2 * half + (k >> 2)) * kBox + 32u * (k & 3), 16u, 1024u);
            const uint64_t bd = sdesc_sw128(b_base + 2048u * k, kBox, 1024u);
            mma_bf16_ss_pair(tmem + kTmemO, ad, bd, idesc2, (i | half | k) != 0 ? 1u : 0u);
          }
          mma_commit_mc(&sm.empty[stage], pair_mask);
          advance();
        }
        // this pair is done reading dS of block i: tell every CTA of the cluster
        mma_commit_mc(&sm.ds_free[db], all_mask);
      };
      int u = 0;
      for (int j = 0; j < nt && ok; ++j) {
        if (owned(j)) {
          if (!mbar_wait_cluster(&sm.s_empty, (u & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < p.num_kb; ++kb) {
            if (!mbar_wait(&sm.full[stage], phase, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sm.stage[stage]);
            const uint32_t b_base = a_base + kBox;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_ss_pair(tmem + kTmemS, sdesc_sw128(a_base + 32u * k, 16u, 1024u),
                               sdesc_sw128(b_base + 32u * k, 16u, 1024u), idesc1, (kb | k) != 0 ? 1u : 0u);
            mma_commit_mc(&sm.empty[stage], pair_mask);
            advance();
          }
          if (!ok) break;
          mma_commit_mc(&sm.s_full, pair_mask);
          ++u;
        }
        if (j >= 1) gemm2(j - 1);
      }
      if (ok) gemm2(nt - 1);
      if (ok) mma_commit_mc(&sm.o_full, pair_mask);
      mma_commit_mc(&sm.drain, pair_mask);
      mbar_wait_drain(&sm.drain, 0);
    }
  } else {
    // ---------------------------------------------------------------------------- epilogue warps
    const int qq = warp & 3;               // TMEM lane quarter
    const int hh = warp >> 2;              // which 128-column half of the 256-wide block
    const int rl = qq * 32 + lane;
    const int row = r0 + rl;
    const float scale = *p.scale;
    const uint32_t s_empty_c = mapa_shared(smem_u32(&sm.s_empty), lead_rank);
    uint32_t ds_full_c[kDsBuf];
    for (int b = 0; b < kDsBuf; ++b) ds_full_c[b] = mapa_shared(smem_u32(&sm.ds_full[b]), lead_rank);
    float row_lse2 = 0.f, row_zf = 0.f, row_coef = 0.f, row_bias2 = 0.f;
    int row_y = -1;
    if (!kVocabRows) {
      if (row < p.BT) {
        const float4 st = p.stats[row];
        row_lse2 = st.x;
        row_zf = st.y;              // valid * (1 + 2 z_loss LSE)
        row_coef = st.z * scale;    // s * valid
        row_y = __float_as_int(st.w);
      }
    } else {
      if (p.bias != nullptr && row < p.V) row_bias2 = __ldg(p.bias + row) * kLog2e;
    }
    float gbias = 0.f;
    bool ok = true;
    const uint32_t ds_row_off = static_cast<uint32_t>(2 * hh) * kBox + static_cast<uint32_t>(rl) * 128u;
    int u = 0;
    int v[kDsBuf] = {};    // blocks received so far into each dS buffer
    for (int j = 0; j < nt && ok; ++j) {
      const int db = j % kDsBuf;
      if (!owned(j)) {
        // block computed by another pair: its dS arrives by bulk copy into this CTA's buffer
        if (warp == 0 && lane == 0) {
          mbar_arrive_expect_tx(&sm.rx_full[db], kDsBytes);
          if (!mbar_wait(&sm.rx_full[db], v[db] & 1, abort)) {
            ok = false;
          } else {
            mbar_arrive_cluster(ds_full_c[db]);
          }
        }
        ++v[db];
        continue;
      }
      if (!mbar_wait(&sm.s_full, u & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[128];
      {
        const uint32_t taddr = tmem + (static_cast<uint32_t>(qq * 32) << 16) + kTmemS + static_cast<uint32_t>(hh * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32cols(taddr + 32u * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(s_empty_c);
      const int sb = u & 1;
      if (kVocabRows && !mbar_wait(&sm.st_full[sb], (u >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const float4* tstats = sm.colstats[kVocabRows ? sb : 0] + (kVocabRows ? hh * 128 : 0);
      const int col0 = j * kPN + hh * 128;
      // every pair must be done with this buffer's previous block before this CTA overwrites it
      if (!mbar_wait_cluster(&sm.ds_free[db], ((j / kDsBuf) & 1) ^ 1, abort)) {
        ok = false;
        break;
      }
      uint8_t* const ds_row = sm.ds[db] + ds_row_off;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint32_t packed[4];
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          float d[2];
#pragma unroll
          for (int w2 = 0; w2 < 2; ++w2) {
            const int i = 8 * ch + 2 * i2 + w2;
            const int col = col0 + i;
            const float sv = __uint_as_float(r[i]);
            float g;
            if (!kVocabRows) {
              const float b2 = (p.bias != nullptr && col < p.V) ? __ldg(p.bias + col) * kLog2e : 0.f;
              const float e = ex2_approx(fmaf(sv, kLog2e, b2 - row_lse2)) * row_zf;
              g = row_coef * (col == row_y ? e - 1.0f : e);
            } else {
              const float4 st = tstats[i];
              const float e = ex2_approx(fmaf(sv, kLog2e, row_bias2 - st.x)) * st.y;
              g = (st.z * scale) * (__float_as_int(st.w) == row ? e - 1.0f : e);
              gbias += g;
            }
            d[w2] = g;
          }
          packed[i2] = pack_bf16x2(d[0], d[1]);
        }
        uint8_t* dst = ds_row + static_cast<uint32_t>(ch >> 3) * kBox;
        const int c = ch & 7;
        *reinterpret_cast<uint4*>(dst + ((c ^ (rl & 7)) << 4)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
      if (kVocabRows) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.st_empty[sb]);
      }
      fence_proxy_async_smem();
      named_barrier_sync(1, kEpiWarps * 32);
      if (warp == 0 && lane == 0) {
        for (int pp = 0; pp < P; ++pp) {
          if (pp == pr) continue;
          const uint32_t dst_rank = static_cast<uint32_t>(2 * pp) + q;
          bulk_copy_to_peer(mapa_shared(smem_u32(sm.ds[db]), dst_rank), sm.ds[db], kDsBytes,
                            mapa_shared(smem_u32(&sm.rx_full[db]), dst_rank));
        }
        mbar_arrive_cluster(ds_full_c[db]);
      }
      ++u;
    }

    if (ok && mbar_wait(&sm.o_full, 0, abort)) {
      tc_fence_after();
      const int n_chunks = (hc + 31) / 32;
      for (int c = hh; c < n_chunks; c += 2) {
        uint32_t vv[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(qq * 32) << 16) + kTmemO + 32u * c, vv);
        tmem_wait_ld();
        const int cb = 32 * c;
        if (!kVocabRows) {
          if (row < p.BT) {
            uint16_t* out = p.grad_input + static_cast<size_t>(row) * p.H + h0 + cb;
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              if (cb + 8 * g8 + 8 <= hc) {
                *reinterpret_cast<uint4*>(out + 8 * g8) =
                    make_uint4(pack_bf16x2(__uint_as_float(vv[8 * g8 + 0]), __uint_as_float(vv[8 * g8 + 1])),
                               pack_bf16x2(__uint_as_float(vv[8 * g8 + 2]), __uint_as_float(vv[8 * g8 + 3])),
                               pack_bf16x2(__uint_as_float(vv[8 * g8 + 4]), __uint_as_float(vv[8 * g8 + 5])),
                               pack_bf16x2(__uint_as_float(vv[8 * g8 + 6]), __uint_as_float(vv[8 * g8 + 7])));
              }
            }
          }
        } else {
          if (row < p.V && p.grad_W != nullptr) {
            float* out = p.grad_W + static_cast<size_t>(row) * p.H + h0 + cb;
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
              if (cb + 4 * g4 + 4 <= hc)
                *reinterpret_cast<float4*>(out + 4 * g4) =
                    make_float4(__uint_as_float(vv[4 * g4 + 0]), __uint_as_float(vv[4 * g4 + 1]),
                                __uint_as_float(vv[4 * g4 + 2]), __uint_as_float(vv[4 * g4 + 3]));
            }
          }
        }
      }
    }
    if (kVocabRows) {
      // this CTA's share of grad_bias (its owned blocks) -> pair 0's CTA with the same rows
      if (hh == 1) sm.half_bias[rl] = gbias;
      named_barrier_sync(1, kEpiWarps * 32);
      if (hh == 0) st_shared_cluster_f32(mapa_shared(smem_u32(&sm.gb_gather[pr][rl]), q), gbias + sm.half_bias[rl]);
    }
  }

  tc_fence_before();
  cluster_sync();
  if (kVocabRows && pr == 0 && warp < 4 && blockIdx.y == 0 && p.grad_bias != nullptr && !sm.abort) {
    const int rl = warp * 32 + lane;
    const int row = r0 + rl;
    if (row < p.V) {
      float acc = 0.f;
      for (int pp = 0; pp < P; ++pp) acc += sm.gb_gather[pp][rl];
      p.grad_bias[row] = acc;
    }
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) atomicOr(status, kStatusTimeout);
}

// Pairs per cluster: the largest of 4, 3, 2, 1 that divides the number of 256-wide H chunks.
int pairs_per_cluster(int h_chunks) {
  for (int P = kMaxPairs; P > 1; --P)
    if (h_chunks % P == 0) return P;
  return 1;
}

}  // namespace

template <bool kVocabRows>
cudaError_t launch_dgrad_pair(const CUtensorMap& rows, const CUtensorMap& cols, const DgPairArgs& a,
                              cudaStream_t stream) {
  PairParams p{};
  p.bias = a.bias;
  p.stats = a.stats;
  p.scale = a.scale;
  p.BT = a.BT;
  p.V = a.V;
  p.H = a.H;
  p.n_rows = kVocabRows ? a.V : a.BT;
  p.n_cols = kVocabRows ? a.BT : a.V;
  p.num_kb = (a.H + kBK - 1) / kBK;
  p.grad_input = a.grad_input;
  p.grad_W = a.grad_W;
  p.grad_bias = a.grad_bias;
  // with only grad_bias requested one H chunk suffices (the GEMM2 result is not stored)
  const int h_chunks = (kVocabRows && p.grad_W == nullptr) ? 1 : (p.H + kHc - 1) / kHc;
  p.P = pairs_per_cluster(h_chunks);
  constexpr size_t smem = pair_smem_bytes<kVocabRows>();
  cudaError_t e = cudaFuncSetAttribute(dgrad_pair_kernel<kVocabRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int row_pairs = (p.n_rows + 2 * kTileM - 1) / (2 * kTileM);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.P * row_pairs, h_chunks / p.P, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * p.P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, dgrad_pair_kernel<kVocabRows>, rows, cols, p, a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template cudaError_t launch_dgrad_pair<false>(const CUtensorMap&, const CUtensorMap&, const DgPairArgs&, cudaStream_t);
template cudaError_t launch_dgrad_pair<true>(const CUtensorMap&, const CUtensorMap&, const DgPairArgs&, cudaStream_t);

}  // namespace flce
