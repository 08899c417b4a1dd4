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
//               K-major layout of the next MMA's A operand; each epilogue warp hands its 32 rows to
//               the same buffer of the other P-1 pairs' CTAs by cp.async.bulk copies between shared
//               memories; never through HBM.  (Stores by the threads themselves, st.shared::cluster,
//               measured about four times slower.)
//     and every pair accumulates its own H chunk:
//       GEMM2   O[256, 256] += dS[256, 256] . cols[256, chunk]      (TMEM, 256 columns, fp32)
//     So the logits of each (row block, column block) are computed ceil(H / (256 P)) times instead of
//     ceil(H / 256) times.
//   * Issue order of a pair's tensor-core work, in steps s = -2P .. n_blocks-1:
//       step s:  GEMM2 of block s (two 128-column halves), then 1/P of the k-blocks of GEMM1 of the
//                pair's own block in [s+P+1, s+2P]
//     so every step carries the same amount of work, and the logits of block j are complete P steps
//     before any pair needs dS of block j: the owner's epilogue computes dS early, stores and sends
//     it as soon as block j-1 has left the dS slots, and the copies overlap the GEMM1 share of step
//     j-1.
//   * The dS buffer holds one block as two half slots.  Every pair's GEMM2 of half h of block j
//     commits on "ds_free[h]" of the pair that writes block j+1 (its owner), and only there, so each
//     ds_free barrier completes exactly one phase per block its CTA writes: the owner's parity waits
//     can never be two phases behind or ahead.
//   * grad_bias (vocabulary rows) is each CTA's fp32 row sum of dS over the blocks it owns, gathered
//     across the pairs in distributed shared memory and added in pair order (deterministic).
//   * Online form of the grad_input pass (dgrad_online_kernel): no row statistics beforehand.  The tile
//     carries P = 2^(z log2 e - ref) against a per-row reference fixed by the first block (the same in
//     every pair, so the accumulators share one scale and nothing is rescaled; "Fused Linear
//     Cross-Entropy", "Strategy 2" keeps a running max instead), the target column is left out of O, the
//     owners keep the row sums and the target logit, and at the end the pairs combine them into the LSE,
//     the statistics and loss terms the rest of the call needs, and grad_input = G u (f O / L + (f p_y - 1)
//     W[y]).  Rows whose sums leave the safe range are left to the classic passes.
//   * Work units: a 1-D grid of clusters, row pair x H group.  When they do not fill their last wave, the
//     row pairs of that wave are split over column ranges (the vocabulary in the grad_input pass, the
//     tokens in the grad_W pass), one cluster per range, and the partial results of those clusters are
//     combined by online_vmerge_kernel / dw_vmerge_kernel.
// All waits are bounded; a wait that gives up flags the status word and the kernel winds down.
#include <algorithm>
#include <type_traits>

#include "flce_kernels.cuh"
#include "sm100.cuh"

namespace flce {

namespace {

constexpr int kPN = 256;                      // logits tile columns = K of GEMM2 per block
constexpr int kBK = 64;
constexpr int kHc = 256;                      // H columns per pair (GEMM2 N)
constexpr int kMaxPairs = 4;                  // pairs per cluster that share each logits tile
// Pairs per side cluster (persistent scheduling, launch_corun): beside four-pair main clusters 2 (4-CTA
// clusters, a row block's logits once per two H chunks; measured at the long workload: 78.3-78.8 ms per
// step with single pairs, 75.4-75.8 with two).  (A side pair must meet whole owner classes of the main
// launch: its blocks j = pr + S t fall in classes j mod P, so S divides P; beside two- or three-pair main
// clusters it would be 1.)
constexpr int side_pairs_for(int P) { return P == 4 ? 2 : 1; }
// Gradient filter: ring of per-block skip verdicts.  The owner of block b publishes them once the logits
// of b are complete, which (in the issue order below) is after every pair finished GEMM2 of block
// b - P - 2, so a ring of more than P + 2 blocks is never overwritten before every CTA has read it.
constexpr int kFlagRing = 8;
static_assert(kFlagRing >= kMaxPairs + 2, "the skip-verdict ring must outlast P + 2 blocks");
constexpr uint32_t kBox = kTileM * kBK * 2;   // 16 KiB: a 128-row x 64-column bf16 box
constexpr uint32_t kStage = 2 * kBox;
constexpr uint32_t kHalfBytes = 2 * kBox;     // one 128-column half of a dS block (per CTA)
constexpr uint32_t kDsBytes = 2 * kHalfBytes;
// grad_W drain: each epilogue warp stages 32 rows of 512 bytes in the operand stages and dS slots, 16
// bytes apart so that the lanes' 16-byte stores meet the fewest bank conflicts
constexpr uint32_t kDrainRowBytes = 512 + 16;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kRecvWarp = 10;
constexpr int kThreads = 11 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;

// Shared memory per CTA: an operand ring of 32 KiB stages, the dS block (two 32 KiB half slots) and, in the
// grad_W pass, one slot with the per-token statistics of the owned block whose dS the epilogue computes
// next (loaded by the producer with that block's last GEMM1 share): the (exponent constant, target) pairs,
// 2 KiB, in the exact pass; the four-word statistics, 4 KiB, in the filtering pass, which also keeps a
// ring of skip verdicts and has one stage fewer (4).  The other passes have 5 stages.  After the main
// loop the dS block gathers the grad_bias partials.
template <bool kVocabRows, bool kFilter, int kSlots = 2>
struct PairCfg {
  static_assert(kSlots == 2 || ((kSlots == 3 || kSlots == 4) && !kFilter), "dS slots: 2, or 3-4 for the exact passes");
  static constexpr int kStages = kSlots == 4 ? 3 : kSlots == 3 ? 4 : (kVocabRows && kFilter) ? 4 : 5;
  static constexpr int kStatCols = kVocabRows ? kPN : 1;
  static constexpr int kRing = kFilter ? kFlagRing : 1;
  using Stat = typename std::conditional<kFilter, float4, float2>::type;
};

template <bool kVocabRows, bool kFilter, int kSlots = 2>
struct PairSmem {
  using Cfg = PairCfg<kVocabRows, kFilter, kSlots>;
  uint8_t stage[Cfg::kStages][kStage];
  uint8_t ds[kSlots][kHalfBytes];
  typename Cfg::Stat colstats[Cfg::kStatCols];
  uint64_t full[Cfg::kStages];
  uint64_t empty[Cfg::kStages];
  uint64_t st_full;
  uint64_t st_empty;
  uint64_t s_full;
  uint64_t s_empty;
  uint64_t ds_full[kSlots];
  uint64_t ds_free[kSlots][kMaxPairs];   // [slot][pair that consumed the slot's previous content]
  uint64_t rx_full[kSlots];
  uint64_t o_full;
  uint64_t o_zero;
  uint64_t drain;
  uint64_t never;             // test-only stall (debug_stall_us): a phase nothing completes
  uint64_t mref_ready;        // online grad_input pass: the per-row reference is in
  uint64_t part_ready;        // online grad_input pass: every pair's per-row partial sums are in
  uint64_t flag_full[Cfg::kRing][2];  // filter: the 8 owner warps' verdicts of [block mod ring][half] are in
  uint32_t skipf[Cfg::kRing][2][8];   // filter: [block mod ring][half][4 x owner CTA + warp] 1 = all small
  uint32_t tmem_base;
  int abort;
  int claim;                  // persistent clusters: the unit CTA 0 claimed for the whole cluster (-1: none)
  // persistent clusters, CTA 0 only, one thread at a time between cluster barriers (claim_next; kept here
  // so that nothing stays live across the unit body): its last claim, the next one-chunk part of it
  // (single-pair clusters), whether the cluster took a unit
  int q_unit, q_sub, q_took;
};
constexpr size_t kSmemBudget = 232448;
// The stage ring and the dS block need 1024-byte alignment (128-byte swizzle atoms).  A layout that fits
// with 1023 bytes of slack is placed at the next 1024-byte boundary; the exact grad_W pass's layout does
// not fit with the slack, so it is placed at the start of the dynamic shared memory, which the kernel
// checks is on a 1024-byte boundary (FLCE_STATUS_INTERNAL and an early return otherwise).
template <bool kVocabRows, bool kFilter, int kSlots = 2>
constexpr size_t pair_smem_slack() {
  return sizeof(PairSmem<kVocabRows, kFilter, kSlots>) + 1024 <= kSmemBudget ? 1024 : 0;
}
template <bool kVocabRows, bool kFilter, int kSlots = 2>
constexpr size_t pair_smem_bytes() {
  return sizeof(PairSmem<kVocabRows, kFilter, kSlots>) + pair_smem_slack<kVocabRows, kFilter, kSlots>();
}
static_assert(pair_smem_bytes<false, false>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<true, false>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<false, true>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<true, true>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<false, false, 4>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<true, false, 4>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<false, false, 3>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(pair_smem_bytes<true, false, 3>() <= kSmemBudget, "shared memory budget of one CTA exceeded");
static_assert(sizeof(float) * kMaxPairs * 2 * kTileM <= kDsBytes, "the dS block gathers the grad_bias partials");
template <bool kVocabRows, bool kFilter, int kSlots>
constexpr bool drain_fits() {
  using S = PairSmem<kVocabRows, kFilter, kSlots>;
  return offsetof(S, ds) == sizeof(S::stage) &&
         sizeof(S::stage) + sizeof(S::ds) >= size_t{kEpiWarps} * 32 * kDrainRowBytes;
}
static_assert(drain_fits<true, false, 2>() && drain_fits<true, true, 2>() && drain_fits<true, false, 4>(),
              "the grad_W drain stages 8 warps x 32 rows in the operand stages and dS slots");

// Gradient filter: the verdict on half `half` of block j, once the 8 epilogue warps of its owner pair that
// hold the half (4 per CTA) have published theirs: 1 = every pair skips it (no operand stage, no MMA, no
// dS hand-over), 0 = keep, -1 = the bounded wait gave up.
template <class Smem>
__device__ __forceinline__ int filter_verdict(Smem& sm, int j, int half, volatile int* abort) {
  const int r = j % kFlagRing;
  if (!mbar_wait_cluster(&sm.flag_full[r][half], static_cast<uint32_t>(j / kFlagRing) & 1u, abort)) return -1;
  const volatile uint32_t* f = sm.skipf[r][half];
  uint32_t all = 1u;
#pragma unroll
  for (int w = 0; w < 8; ++w) all &= f[w];
  return all != 0u ? 1 : 0;
}

struct PairParams {
  const float* bias;
  const float4* stats;
  const float2* stats_ct;   // (x, y) of stats: what the exact grad_W pass stages per block
  const float* colb2;
  const float* scale;
  const uint32_t* zf_neg;
  float z_loss;
  int accumulate;
  float filter_eps;         // > 0: skip GEMM2 of dS halves whose entries are all below it
  uint32_t* skip_count;     // halves skipped (filter statistics)
  const int32_t* row_perm;  // grad_W pass: output row of each vocabulary row (vocabulary sort), or null
  int BT, V, H;
  int n_rows, n_cols, num_kb;
  int P;                    // pairs per cluster
  uint16_t* grad_input;
  float* grad_W;
  float* grad_bias;
  const uint32_t* gate;     // non-null: the launch does nothing unless *gate != 0
  // grad_input pass without a prior LSE pass (online softmax against a fixed per-row reference)
  const int64_t* target;
  int64_t ignore_index;
  const float* grad_tok;    // per-token upstream gradient, or null (ones)
  const uint16_t* Wmat;     // W, for the target-row term
  float* mref_g;            // [BT rounded up to 256] per-row reference, log2 units
  float4* part_g;           // [BT rounded up to 256][kMaxPairs][2]: (sum of 2^(x - ref), z_y or -inf,
                            //  sum of 2^(x - ref) z, 0)
  float* entropy_out;       // per-row entropy of softmax(z), or null
  uint32_t* row_redo;       // online pass: per row, 1 when its sum left the safe range (row not written);
                            // classic grad_input pass behind it: write only those rows
  float4* stats_out;        // per-token statistics for the grad_W pass
  float2* stats_ct_out;     // their compact (x, y) copy
  float* row_loss;
  float* loss_tok;
  uint32_t* zf_neg_out;
  uint32_t* fallback;       // set when a row's sum left the safe range: the classic passes redo the work
  // online pass, vocabulary-split work units (unit su covers column blocks [jb, je) of its 256 rows and
  // writes partial results instead of the row outputs; online_vmerge_kernel combines them):
  float* vs_mref;           // [su][256] the unit's per-row reference
  float4* vs_part;          // [su][256][kMaxPairs][2] its pairs' partial sums (as part_g)
  float4* vs_stat;          // [su][256] (L, z_y or -inf, T, reference) over the unit's columns
  float* vs_o;              // [su][256][P * 256] its unnormalised accumulator O (grad_W pass: its partial
                            // grad_W rows, the units then covering token ranges)
  float* vs_gb;             // grad_W pass: [su][256] partial grad_bias
  uint32_t* vs_count;       // receives the number of split units (workspace header)
  uint32_t debug_stall_us;  // test-only: the producer first waits this long on `never`, then gives up
};

// The block whose GEMM1 pair `pr` works on in step s (the one it owns in [s+P+1, s+2P]) and which
// share (0 .. P-1) of that block's k-blocks belongs to this step.  The logits of block j are then
// complete P steps before GEMM2 of block j, so the owner has time to turn them into dS and send
// them; and the owner's previous block j-P left the dS slots at step j-P-1, before the first share of
// its next GEMM1 (step j-P+1) needs the logits buffer back, so that GEMM1 never waits on a store.
struct G1Share {
  int block;
  int prog;
};
__device__ __forceinline__ G1Share g1_share(int s, int pr, int P) {
  const int lead = P + 1;
  int d = (pr - (s + lead)) % P;
  if (d < 0) d += P;
  return G1Share{s + lead + d, P - 1 - d};
}
__device__ __forceinline__ int share_begin(int prog, int num_kb, int P) { return (prog * num_kb) / P; }

// Row constants of the dS arithmetic of one epilogue thread (G: the gradient scale, u: a token's
// upstream gradient, f = 1 + 2 z_loss LSE).
struct DsRow {
  float c;      // grad_input pass: log2(G u f) - LSE2 (-inf for ignored rows); grad_W pass: b log2 e + log2 G
  float f;      // grad_input pass, general form: f
  float lse2;   // grad_input pass, general form: LSE log2 e
  float coef;   // grad_input pass: G u [valid], the weight of the onehot term
  float bias2;  // grad_W pass, general form: b log2 e
  float scale;  // G
  float zl2;    // 2 z_loss ln 2 (f = 1 + zl2 LSE2)
  int y;        // grad_input pass: target column (-1 if none); grad_W pass: this row's vocabulary index
};

// Per-token statistics of the grad_W pass's columns: the staged (x, y) pairs of the exact pass (the other
// two words from global memory, where needed: the rare target column and the general form), or the staged
// four words of the filtering pass.
__device__ __forceinline__ float2 stat_xy(const float2& s) { return s; }
__device__ __forceinline__ float2 stat_xy(const float4& s) { return make_float2(s.x, s.y); }
__device__ __forceinline__ float4 stat_full(const float2* /*staged*/, const float4* __restrict__ g, int i) {
  return __ldg(g + i);
}
__device__ __forceinline__ float4 stat_full(const float4* s, const float4* /*global*/, int i) { return s[i]; }

// dS of 64 consecutive logits of one row, in place (fp32 bits in, fp32 bits out).
//   grad_input pass (rows = tokens): columns col0.. are vocabulary entries; colb2 holds the bias in
//     log2 units (-inf past V); `plain` means no bias and no column past V in this chunk.
//   grad_W pass (rows = vocabulary): columns are tokens; tstats holds their staged statistics, gst the
//     same columns' four-word statistics in global memory.
//   fge > 0 (gradient filter, grad_W pass): fover is set when some |dS| exceeds fge |w| (w the column's
//   gradient weight), checked where each column's statistics are loaded anyway.
template <bool kVocabRows, class St>
__device__ __forceinline__ void ds_chunk64(uint32_t (&r)[64], int col0, const DsRow& rc, bool general, bool plain,
                                           const float* __restrict__ colb2, const St* tstats,
                                           const float4* __restrict__ gst, float& gbias, float fge = 0.f,
                                           int* fover = nullptr) {
  if (!kVocabRows) {
    if (general) {
#pragma unroll
      for (int i4 = 0; i4 < 16; ++i4) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(colb2 + col0) + i4);
        const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 4 * i4 + k;
          const float e = ex2_approx(fmaf(__uint_as_float(r[i]), kLog2e, bb[k] - rc.lse2)) * rc.f;
          r[i] = __float_as_uint(rc.coef * (col0 + i == rc.y ? e - 1.0f : e));
        }
      }
      return;
    }
    if (plain) {
#pragma unroll
      for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[i]), kLog2e, rc.c)));
    } else {
#pragma unroll
      for (int i4 = 0; i4 < 16; ++i4) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(colb2 + col0) + i4);
        r[4 * i4 + 0] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[4 * i4 + 0]), kLog2e, rc.c + b.x)));
        r[4 * i4 + 1] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[4 * i4 + 1]), kLog2e, rc.c + b.y)));
        r[4 * i4 + 2] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[4 * i4 + 2]), kLog2e, rc.c + b.z)));
        r[4 * i4 + 3] = __float_as_uint(ex2_approx(fmaf(__uint_as_float(r[4 * i4 + 3]), kLog2e, rc.c + b.w)));
      }
    }
    if (static_cast<unsigned>(rc.y - col0) < 64u) {
      // the target column lies in this chunk (rare): subtract the onehot weight there
#pragma unroll
      for (int i = 0; i < 64; ++i)
        if (col0 + i == rc.y) r[i] = __float_as_uint(__uint_as_float(r[i]) - rc.coef);
    }
  } else {
    if (general) {
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float4 st = stat_full(tstats, gst, i);
        const int yt = __float_as_int(st.y);
        const float e = ex2_approx(fmaf(__uint_as_float(r[i]), kLog2e, rc.bias2 - st.w)) * fmaf(rc.zl2, st.w, 1.0f);
        const float g = (rc.scale * st.z) * (yt == rc.y ? e - 1.0f : e);
        gbias += g;
        if (fover != nullptr) *fover |= fabsf(g) > fge * fabsf(st.z) ? 1 : 0;
        r[i] = __float_as_uint(g);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        // (exponent constant and target of the token; its gradient weight only where needed)
        const float2 st = stat_xy(tstats[i]);
        float g = ex2_approx(fmaf(__uint_as_float(r[i]), kLog2e, rc.c + st.x));
        if (__float_as_int(st.y) == rc.y) g -= rc.scale * stat_full(tstats, gst, i).z;
        gbias += g;
        if (fover != nullptr) *fover |= fabsf(g) > fge * fabsf(stat_full(tstats, gst, i).z) ? 1 : 0;
        r[i] = __float_as_uint(g);
      }
    }
  }
}

// Gradient filter, grad_input pass: true when every one of this row's 64 dS values (fp32 bits) is small
// relative to the row's gradient weight, |dS| <= eps |G u [valid]| (zero-weight rows are all zero).
__device__ __forceinline__ bool filter_small_row(const uint32_t (&r)[64], const DsRow& rc, float eps) {
  float worst = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) worst = fmaxf(worst, fabsf(__uint_as_float(r[i])));
  return worst <= eps * fabsf(rc.coef);
}

// Online grad_input pass: 64 consecutive logits of one row (fp32 bits in) -> 2^(S log2 e + b log2 e - ref)
// (fp32 bits out), with c = -ref, and their sum added to lsum (with ent, the sum of each times its logit
// z = S + b to tsum); the target column's logit (+ bias) goes to zy and its entry to 0 (its gradient term
// is added exactly at the end; it stays in the sums).
__device__ __forceinline__ void online_chunk64(uint32_t (&r)[64], int col0, float c, bool plain,
                                               const float* __restrict__ colb2, const float* __restrict__ bias, int y,
                                               float& lsum, float& zy, bool ent, float& tsum) {
  const bool has_y = static_cast<unsigned>(y - col0) < 64u;
  if (has_y) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (col0 + i == y) zy = __uint_as_float(r[i]) + (bias != nullptr ? __ldg(bias + y) : 0.f);
  }
  float sum = 0.f, tz = 0.f;
  if (plain) {
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float z = __uint_as_float(r[i]);
      const float v = ex2_approx(fmaf(z, kLog2e, c));
      r[i] = __float_as_uint(v);
      sum += v;
      if (ent) tz = fmaf(v, z, tz);
    }
  } else {
#pragma unroll
    for (int i4 = 0; i4 < 16; ++i4) {
      const float4 b = __ldg(reinterpret_cast<const float4*>(colb2 + col0) + i4);
      const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float z = __uint_as_float(r[4 * i4 + k]);
        const float v = ex2_approx(fmaf(z, kLog2e, c + bb[k]));
        r[4 * i4 + k] = __float_as_uint(v);
        sum += v;
        // (columns past V carry b = -inf and v = 0: no term)
        if (ent && bb[k] != -INFINITY) tz = fmaf(v, fmaf(bb[k], kLn2, z), tz);
      }
    }
  }
  if (ent) tsum += tz;
  if (has_y) {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (col0 + i == y) r[i] = 0u;
  }
  lsum += sum;
}

// Online grad_input pass: one row's outputs from its sums over the whole vocabulary against the reference
// ref (log2 units): L = sum_n 2^(z_n log2 e - ref), zy = the target logit (-inf if none), T = sum_n
// 2^(z_n log2 e - ref) z_n.  With `write` (one thread per row) stores the loss terms, the statistics the
// grad_W pass reads, zf_neg, the entropy and the redo flag.  Returns the coefficients of
// grad_input[row] = c1 O[row] + c2 W[y] and whether the row is in the safe range:
//   LSE = (ref + log2 L) ln 2, f = 1 + 2 z_loss LSE, c1 = G u f / L (O holds sum over n != y of
//   2^(..) W[n]), c2 = G u (f p_y - 1).
struct OnlineRow {
  float c1, c2;
  bool ok;
};
__device__ __forceinline__ OnlineRow online_row_finish(const PairParams& p, int row, float ref, float L, float zy,
                                                       float T, int y, float u, float scale, bool write) {
  OnlineRow r{0.f, 0.f, true};
  const float lse2 = ref + log2f(L);
  const float lse = lse2 * kLn2;
  const bool valid = y >= 0;
  const float f = 1.0f + 2.0f * p.z_loss * lse;
  if (valid) {
    r.c1 = scale * u * f / L;
    r.c2 = scale * u * (f * ex2_approx(fmaf(zy, kLog2e, -lse2)) - 1.0f);
  }
  // 2^115 leaves room for the accumulator's sums over the vocabulary; beyond it (or for a sum that is
  // not finite) the row is left unwritten and the classic passes redo it
  r.ok = L < 0x1p115f;
  if (write && row < p.BT) {
    const float lt = valid ? (lse - zy) + p.z_loss * lse * lse : 0.f;
    p.row_loss[row] = lt;
    if (p.loss_tok != nullptr) p.loss_tok[row] = lt;
    const float uf = u * f;
    if (valid && u != 0.f && !(uf > 0.f)) atomicOr(p.zf_neg_out, 1u);
    const float2 ct = make_float2(valid && uf > 0.f ? log2f(uf) - lse2 : -INFINITY, __int_as_float(valid ? y : -1));
    p.stats_out[row] = make_float4(ct.x, ct.y, valid ? u : 0.f, lse2);
    p.stats_ct_out[row] = ct;
    // entropy of softmax(z) = LSE - sum_n p_n z_n, for every row
    if (p.entropy_out != nullptr) p.entropy_out[row] = lse - T / L;
    p.row_redo[row] = r.ok ? 0u : 1u;
    if (!r.ok) atomicOr(p.fallback, 1u);
  }
  return r;
}

// The shared-memory layout of this CTA (PairSmem), or null when a layout without slack does not start on
// the 1024-byte boundary it needs (every CTA of a launch sees the same offset).
template <bool kVocabRows, bool kFilter, int kSlots>
__device__ __forceinline__ PairSmem<kVocabRows, kFilter, kSlots>* pair_smem_of() {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uintptr_t base = reinterpret_cast<uintptr_t>(smem_raw);
  if (pair_smem_slack<kVocabRows, kFilter, kSlots>() != 0) {
    base = (base + 1023) & ~uintptr_t(1023);
  } else if ((smem_u32(smem_raw) & 1023u) != 0u) {
    return nullptr;
  }
  return reinterpret_cast<PairSmem<kVocabRows, kFilter, kSlots>*>(base);
}

// Work queue of a pass run by persistent clusters (word != null): the main launch's clusters of four
// pairs take whole units (row pair x H group) from the bottom of the row pairs; a second launch of
// side clusters of S pairs (the side launch, on the SMs the main launch leaves idle; S = side_pairs_for(P))
// takes units of one row pair and S 256-wide H chunks from the top, computing that row pair's logits once
// per S chunks; a third launch of single-pair clusters (on the SMs where no side cluster finds room) takes
// the same units as the side launch, from the same count, and runs each as S one-chunk units in turn,
// computing the logits once per chunk.  One 64-bit word holds both counts (main units claimed | side
// units claimed << 32), so that a row pair is never split between the main launch and the others.  The
// side clusters open a new row pair only while the main launch has at least `reserve` row pairs left:
// enough to keep it busy while they finish that row pair.  The single-pair clusters take any unit, also
// one that continues a row pair a side cluster began, only with their own (larger) reserve to spare, and
// stop at the first they cannot take.
enum : int { kRoleMain = 1, kRoleSide = 2, kRoleSingle = 3 };
struct WorkQueue {
  unsigned long long* word;   // zeroed before the pass; null: one cluster per unit (blockIdx), no queue
  uint32_t* side_count;       // [2] side launches that ran, side clusters that took a unit (workspace
                              // header), or null
  uint32_t* single_count;     // [2] the same for the single-pair launches, or null
  uint32_t* single_units;     // this pass's units taken by single-pair clusters, or null
  int role;
  int row_pairs;
  int main_groups;            // H groups per row pair of a main unit (h_chunks / 4)
  int side_groups;            // H groups per row pair of a side unit (h_chunks / S)
  int side_chunks;            // S: H chunks per side unit
  int reserve;
};

// The next unit for this launch's role, -1 when there is none left for it, -2 when the compare-and-swap
// did not settle (the caller flags the status; with a few dozen clusters claiming every few hundred
// microseconds it always settles at once).
__device__ __forceinline__ int claim_unit(const WorkQueue& q) {
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(q.word);
  for (int tries = 0; tries < (1 << 16); ++tries) {
    const int a = static_cast<int>(cur & 0xffffffffull);
    const int b = static_cast<int>(cur >> 32);
    const int a_rows = (a + q.main_groups - 1) / q.main_groups;   // row pairs the main launch has begun
    const int b_rows = (b + q.side_groups - 1) / q.side_groups;   // row pairs the side launch has begun
    unsigned long long next;
    if (q.role == kRoleMain) {
      if (a / q.main_groups >= q.row_pairs - b_rows) return -1;
      next = cur + 1ull;
    } else {
      // (side: a row pair already begun is always finished, a new one only with `reserve` row pairs to
      // spare; single-pair: every unit only with its reserve to spare, which is at least the side's, so
      // that a side cluster is always there to finish a row pair it began)
      const bool check = q.role == kRoleSingle || b % q.side_groups == 0;
      if (check && (q.row_pairs - 1 - b / q.side_groups) - a_rows < q.reserve) return -1;
      next = cur + (1ull << 32);
    }
    const unsigned long long seen = atomicCAS(q.word, cur, next);
    if (seen == cur) return q.role == kRoleMain ? a : b;
    cur = seen;
  }
  return -2;
}

// Rank 0's claim of its cluster's next unit, handed to every CTA of the cluster (sm.claim) as
// claim x n_sub + part, or -1 for none: once by thread 0 before the first unit, then by the MMA issuer of
// each unit once its last MMA has completed, so that the claim's atomic overlaps the unit's accumulator
// drain; every CTA reads it after the unit's last cluster barrier.  A single-pair cluster runs each side
// unit it claims as n_sub = side_chunks one-chunk units in turn.  Nothing more is claimed once the pass's
// status holds a timeout or (check_abort) a CTA of the cluster gave up on a wait in this unit.  The state
// (q_unit, q_sub, q_took) lives in rank 0's shared memory, touched by one thread between cluster barriers.
template <class Smem>
__device__ __forceinline__ void claim_next(Smem& sm, const WorkQueue& wq, uint32_t* status, int n_ctas,
                                           bool check_abort) {
  const int n_sub = wq.role == kRoleSingle ? wq.side_chunks : 1;
  const int sub = sm.q_sub;
  if (sub == 0) {
    bool stop = (*reinterpret_cast<volatile uint32_t*>(status) & kStatusTimeout) != 0u;
    for (int r = 0; r < n_ctas && check_abort && !stop; ++r)
      stop = ld_shared_cluster_u32(mapa_shared(smem_u32(&sm.abort), static_cast<uint32_t>(r))) != 0u;
    int cl = stop ? -1 : claim_unit(wq);
    if (cl == -2) {
      atomicOr(status, kStatusInternal);
      cl = -1;
    }
    uint32_t* const counts = wq.role == kRoleSide ? wq.side_count : wq.role == kRoleSingle ? wq.single_count : nullptr;
    if (cl >= 0 && !sm.q_took && counts != nullptr) atomicAdd(counts + 1, 1u);
    if (cl >= 0 && wq.role == kRoleSingle && wq.single_units != nullptr) atomicAdd(wq.single_units, 1u);
    if (cl >= 0) sm.q_took = 1;
    sm.q_unit = cl;
  }
  sm.q_sub = sub + 1 == n_sub ? 0 : sub + 1;
  const int v = sm.q_unit < 0 ? -1 : sm.q_unit * n_sub + sub;
  for (int r = 0; r < n_ctas; ++r)
    st_shared_cluster_u32(mapa_shared(smem_u32(&sm.claim), static_cast<uint32_t>(r)), static_cast<uint32_t>(v));
}

// TMEM of a dgrad_pair_body call: allocated and freed by it (one unit per CTA), or held by the caller
// across the units of a persistent CTA.  (Allocating inside the body keeps the one-unit kernels' register
// allocation as it was.)
enum : int { kTmemOneUnit = 0, kTmemHeld = 1 };

// kOwn = A > 1 in dgrad_pair_body: a pair of a cluster of P = 4 / A pairs keeps A running sums, one per
// owner class of a four-pair cluster it meets (its t-th block, j = pr + t P, belongs to class
// j mod 4 = pr + (t mod A) P), rotating them so that a0 always holds the current block's.  After its n_own blocks, a_i holds
// slot (n_own - 1 + i) mod A; slot_sum returns slot s.  A slot that met no block holds 0.
__device__ __forceinline__ float slot_sum(float a0, float a1, float a2, float a3, int s, int n_own, int A) {
  const int i = (((s - (n_own - 1)) % A) + A) % A;
  return i == 0 ? a0 : i == 1 ? a1 : i == 2 ? a2 : a3;
}

// kFilter: the gradient-filtering variant (a separate instantiation, so the exact path carries none of
// its checks).
// One cluster's work: rows [256 row_pair, +256) (128 per CTA of each pair) and the H chunks of
// group hgroup (P consecutive 256-wide chunks, one per pair).
// Columns: blocks [jb, je) of 256 (all of them except for a vocabulary-split unit of the online pass, su >= 0).
// kOwn = 2 or 4: a cluster of two pairs or one pair standing in for a cluster of four pairs, whose results
// it reproduces bit for bit: the per-row sums that four pairs would keep apart (each over the blocks it
// owns, j mod 4) are kept apart too (kOwn of them per pair) and combined in the same order (the online
// pass's softmax sums, grad_bias).  kOwn = 1: no owner classes (P pairs, each keeping one sum).
template <bool kVocabRows, bool kFilter, bool kOnline = false, int kSlots = 2, int kOwn = 1, int kTmem = 0>
__device__ __forceinline__ void dgrad_pair_body(const CUtensorMap& tm_rows, const CUtensorMap& tm_cols,
                                                const PairParams& p, uint32_t* __restrict__ status, int row_pair,
                                                int hgroup, int jb, int je, int su, const WorkQueue& wq) {
  static_assert(!kOnline || (!kVocabRows && !kFilter), "the online form is a grad_input pass without the filter");
  static_assert(kOwn == 1 || ((kOwn == 2 || kOwn == 4) && !kFilter),
                "owner-class sums per pair: 1, or 2 / 4 (two-pair / single-pair clusters) for the exact passes");
  using Smem = PairSmem<kVocabRows, kFilter, kSlots>;
  constexpr int kStages = Smem::Cfg::kStages;
  // (run_units has checked the gate and the layout's alignment and allocated TMEM)
  Smem& sm = *pair_smem_of<kVocabRows, kFilter, kSlots>();
  const uint32_t rank = cluster_ctarank();
  const int P = p.P;
  const int pr = static_cast<int>(rank >> 1);       // pair index within the cluster
  const uint32_t q = rank & 1u;                     // half of the pair (which 128 rows)
  const bool leader = (q == 0);
  const uint32_t lead_rank = rank & ~1u;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << (2 * pr));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r0 = row_pair * (2 * kTileM) + static_cast<int>(q) * kTileM;
  const int h0 = (hgroup * P + pr) * kHc;
  const int hc = min(kHc, p.H - h0);
  const uint32_t n2 = hc > 128 ? 256u : 128u;   // GEMM2 N; columns past H are zero-filled by TMA
  const int nbox2 = static_cast<int>(n2) / 128; // 64-column boxes per CTA per GEMM2 stage
  if (je < 0) je = (p.n_cols + kPN - 1) / kPN;
  const int nt = je - jb;   // column blocks of this unit; j below counts from jb
  const int nkb = p.num_kb;
  constexpr bool filt = kFilter;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    if (kVocabRows) {
      mbar_init(&sm.st_full, 1);
      mbar_init(&sm.st_empty, kEpiWarps);
    }
    for (int b = 0; b < kSlots; ++b) {
      // 8 arrivals per content: the owner pair's 8 epilogue warps (4 per CTA), or 4 from each CTA's receiver
      mbar_init(&sm.ds_full[b], 8);
      for (int pp = 0; pp < kMaxPairs; ++pp) mbar_init(&sm.ds_free[b][pp], 1);
      mbar_init(&sm.rx_full[b], 1);
    }
    if (filt) {
      for (int r = 0; r < kFlagRing; ++r)
        for (int b = 0; b < 2; ++b) mbar_init(&sm.flag_full[r][b], 8);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_empty, 2 * kEpiWarps);
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_zero, 2 * kEpiWarps);
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.never, 1);
    if (kOnline) {
      mbar_init(&sm.mref_ready, 4);       // the 4 warps of pair 0's CTA with these rows that hold half 0
      mbar_init(&sm.part_ready, 8 * P);   // the 8 epilogue warps of every pair's CTA with these rows
    }
    sm.abort = 0;
    fence_mbarrier_init();
  }
  if (kTmem != kTmemHeld && warp == kMmaWarp) {
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
  // grad_W pass: this epilogue thread's grad_bias partial (its row, its half); with kOwn > 1, one per
  // owner-class slot (slot_sum)
  float gbias_out = 0.f, gbias_c1 = 0.f, gbias_c2 = 0.f, gbias_c3 = 0.f;
  // owner classes a pair meets (its cluster has kMaxPairs / kOwn pairs)
  constexpr int n_slots = kOwn;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // test-only (debug_stall_us): wait for a phase that nothing completes, before any copy is issued; the
      // wait gives up like any other and the whole cluster winds down with nothing in flight
      if (p.debug_stall_us != 0u) ok = mbar_wait(&sm.never, 0, abort, 1000ull * p.debug_stall_us);
      int us = 0;   // grad_W pass: owned blocks whose statistics have been loaded
      auto next = [&]() {
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      };
      auto load_gemm2 = [&](int j, int half) {
        if (!ok || j < 0) return;
        if (filt) {
          const int verdict = filter_verdict(sm, j, half, abort);
          if (verdict < 0) {
            ok = false;
            return;
          }
          if (verdict == 1) return;   // skipped by every pair: no operand stage
        }
        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
          ok = false;
          return;
        }
        const uint32_t fb = mapa_shared(smem_u32(&sm.full[stage]), lead_rank);
        if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2u * nbox2 * kBox);
        for (int b = 0; b < nbox2; ++b)
          tma_load_2d_pair(sm.stage[stage] + b * kBox, &tm_cols, fb,
                           h0 + static_cast<int>(q * (n2 / 2)) + 64 * b, (jb + j) * kPN + half * kTileM);
        next();
      };
      for (int s = -2 * P; s < nt && ok; ++s) {
        const G1Share g = g1_share(s, pr, P);
        const bool has_g1 = g.block >= 0 && g.block < nt;
        const int kb0 = has_g1 ? share_begin(g.prog, nkb, P) : 0;
        const int kb1 = has_g1 ? share_begin(g.prog + 1, nkb, P) : 0;
        auto load_stats = [&]() {
          // grad_W pass: the statistics of the owned block whose last GEMM1 share this step loads, into the
          // single slot once the epilogue has turned the previous owned block into dS (stats are padded to a
          // multiple of 256 tokens)
          if (!kVocabRows || !ok || !has_g1 || g.prog != P - 1) return;
          if (!mbar_wait(&sm.st_empty, (us & 1) ^ 1, abort)) {
            ok = false;
            return;
          }
          const size_t col = static_cast<size_t>(jb + g.block) * kPN;
          const void* src = kFilter ? static_cast<const void*>(p.stats + col) : static_cast<const void*>(p.stats_ct + col);
          mbar_arrive_expect_tx(&sm.st_full, static_cast<uint32_t>(sizeof(sm.colstats)));
          bulk_load_1d(sm.colstats, src, static_cast<uint32_t>(sizeof(sm.colstats)), &sm.st_full);
          ++us;
        };
        auto load_gemm1 = [&](int kb_begin, int kb_end) {
          for (int kb = kb_begin; kb < kb_end && ok; ++kb) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
              ok = false;
              return;
            }
            const uint32_t fb = mapa_shared(smem_u32(&sm.full[stage]), lead_rank);
            if (leader) mbar_arrive_expect_tx(&sm.full[stage], 2 * kStage);
            tma_load_2d_pair(sm.stage[stage], &tm_rows, fb, kb * kBK, r0);
            tma_load_2d_pair(sm.stage[stage] + kBox, &tm_cols, fb, kb * kBK,
                             (jb + g.block) * kPN + static_cast<int>(q) * kTileM);
            next();
          }
        };
        // a step's tensor work, in the MMA issuer's order: GEMM2 of half 0 and half 1, then the GEMM1 share
        load_gemm2(s, 0);
        load_gemm2(s, 1);
        load_stats();
        load_gemm1(kb0, kb1);
      }
      if (ok) {
        // every stage's last release (an MMA commit, multicast to both CTAs of the pair) has arrived
        // before the unit ends, so that a persistent cluster can initialise the barriers for its next unit
        for (int s = 0; s < kStages && ok; ++s) {
          ok = mbar_wait(&sm.empty[stage], phase ^ 1u, abort);
          next();
        }
      }
      if (!ok) {
        // let copies already issued land before the CTA can finish
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------------- MMA issuer (even CTA)
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
      auto gemm2 = [&](int j, int half) {
        if (!ok || j < 0) return;
        // content n = 2j + half of the dS slots sits in slot n mod kSlots; the pair that writes that slot's
        // next content (n + kSlots) reuses it once every pair is done with this one
        const int n_ds = 2 * j + half;
        const int slot = n_ds % kSlots;
        const int j_next = (n_ds + kSlots) >> 1;
        const uint16_t next_owner = static_cast<uint16_t>(3u << (2 * (j_next % P)));
        if (filt && j == 0 && half == 0) {
          // with the filter O starts from the epilogue's zeros and every GEMM2 accumulates
          if (!mbar_wait_cluster(&sm.o_zero, 0, abort)) {
            ok = false;
            return;
          }
        }
        {
          // (also for a skipped half: its slot may be rewritten only after anything sent into it landed)
          if (!mbar_wait_cluster(&sm.ds_full[slot], static_cast<uint32_t>(n_ds / kSlots) & 1u, abort)) {
            ok = false;
            return;
          }
          bool skip = false;
          if (filt) {
            const int verdict = filter_verdict(sm, j, half, abort);
            if (verdict < 0) {
              ok = false;
              return;
            }
            skip = verdict == 1;
          }
          if (!skip) {
            if (!mbar_wait(&sm.full[stage], phase, abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sm.ds[slot]);
            const uint32_t b_base = smem_u32(sm.stage[stage]);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ad = sdesc_sw128(a_base + (k >> 2) * kBox + 32u * (k & 3), 16u, 1024u);
              const uint64_t bd = sdesc_sw128(b_base + 2048u * k, kBox, 1024u);
              mma_bf16_ss_pair(tmem + kTmemO, ad, bd, idesc2, (filt || (j | half | k) != 0) ? 1u : 0u);
            }
            mma_commit_mc(&sm.empty[stage], pair_mask);
            advance();
          } else if (p.skip_count != nullptr) {
            atomicAdd(p.skip_count, 1u);
          }
          if (j_next < nt) mma_commit_mc(&sm.ds_free[slot][pr], next_owner);
        }
      };
      int u = 0;   // owned blocks whose GEMM1 has been issued in full
      for (int s = -2 * P; s < nt && ok; ++s) {
        const G1Share g = g1_share(s, pr, P);
        const bool has_g1 = g.block >= 0 && g.block < nt;
        const int kb0 = has_g1 ? share_begin(g.prog, nkb, P) : 0;
        const int kb1 = has_g1 ? share_begin(g.prog + 1, nkb, P) : 0;
        bool first = true;
        auto gemm1 = [&](int kb_begin, int kb_end) {
          if (!ok || !has_g1) return;
          if (first && g.prog == 0) {
            // the epilogue must have read the previous logits tile out of TMEM
            if (!mbar_wait_cluster(&sm.s_empty, (u & 1) ^ 1, abort)) {
              ok = false;
              return;
            }
            tc_fence_after();
          }
          first = false;
          for (int kb = kb_begin; kb < kb_end; ++kb) {
            if (!mbar_wait(&sm.full[stage], phase, abort)) {
              ok = false;
              return;
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
        };
        gemm2(s, 0);
        gemm2(s, 1);
        gemm1(kb0, kb1);
        if (ok && has_g1 && g.prog == P - 1) {
          mma_commit_mc(&sm.s_full, pair_mask);
          ++u;
        }
      }
      if (ok) mma_commit_mc(&sm.o_full, pair_mask);
      mma_commit_mc(&sm.drain, pair_mask);
      mbar_wait_drain(&sm.drain, 0);
      // persistent cluster of the grad_W pass: the next unit's claim, while the epilogue drains the
      // accumulator
      if (kTmem == kTmemHeld && kVocabRows && rank == 0) claim_next(sm, wq, status, 2 * P, true);
    }
  } else if (warp == kRecvWarp) {
    // ---------------------------------------- dS halves of blocks computed by the other pairs
    if (lane == 0 && P > 1) {
      int v = 0;   // blocks received so far
      int recv[kSlots] = {};   // contents received into each slot so far
      bool ok = true;
      for (int j = 0; j < nt && ok; ++j) {
        if (j % P == pr) continue;
        for (int half = 0; half < 2; ++half) {
          const int slot = (2 * j + half) % kSlots;
          mbar_arrive_expect_tx(&sm.rx_full[slot], kHalfBytes);
          if (!mbar_wait_cluster(&sm.rx_full[slot], static_cast<uint32_t>(recv[slot]++) & 1u, abort)) {
            ok = false;
            break;
          }
          // (the half was written by the other pair's stores; order them before the MMAs that read it)
          fence_proxy_async_smem();
          mbar_arrive_cluster_cnt(mapa_shared(smem_u32(&sm.ds_full[slot]), lead_rank), 4);
        }
        ++v;
      }
    }
  } else {
    // ---------------------------------------------------------------------------- epilogue warps
    const int qq = warp & 3;               // TMEM lane quarter
    const int hh = warp >> 2;              // which 128-column half of the 256-wide block
    const int rl = qq * 32 + lane;
    const int row = r0 + rl;
    const float scale = *p.scale;
    const uint32_t s_empty_c = mapa_shared(smem_u32(&sm.s_empty), lead_rank);
    // dS[m, n] = s [m valid] f_m 2^(S log2 e + b_n log2 e - LSE2_m) - s [n = y_m], with f = 1 + 2 z_loss LSE,
    // evaluated as 2^(S log2 e + c) with c = log2(s f) - LSE2 + b log2 e gathered per row or column.
    // When some valid row has f <= 0 (LSE <= -1/(2 z_loss)) the log form does not apply and every tile
    // takes the general form, with f and the onehot weight as separate factors.
    const bool general = !kOnline && (*p.zf_neg != 0u);
    const float log2s = log2f(scale);
    DsRow rc{-INFINITY, 0.f, 0.f, 0.f, 0.f, scale, 2.0f * p.z_loss * kLn2, -1};
    // online form: no statistics yet; this row's target and upstream gradient, its reference (from the first
    // block, once pair 0 has published it), and the running sum / target logit of the columns it owns
    float on_ref = 0.f, on_lsum = 0.f, on_zy = -INFINITY, on_u = 0.f, on_tsum = 0.f;
    const bool on_ent = kOnline && p.entropy_out != nullptr;
    bool on_have_ref = false;
    // where this row's reference and partial sums go (a vocabulary-split unit has its own; rloc = the row
    // within the unit's 256)
    const int rloc = static_cast<int>(q) * kTileM + rl;
    float* const on_mref = !kOnline ? nullptr
                           : su < 0 ? p.mref_g + row
                                    : p.vs_mref + static_cast<size_t>(su) * 256 + rloc;
    float4* const on_part = !kOnline ? nullptr
                            : su < 0 ? p.part_g + static_cast<size_t>(row) * kMaxPairs * 2
                                     : p.vs_part + (static_cast<size_t>(su) * 256 + rloc) * kMaxPairs * 2;
    if (kOnline) {
      if (row < p.BT) {
        const int64_t y = p.target[row];
        rc.y = (y != p.ignore_index && y >= 0 && y < p.V) ? static_cast<int>(y) : -1;
        on_u = p.grad_tok != nullptr ? p.grad_tok[row] : 1.0f;
      }
    } else if (!kVocabRows) {
      if (row < p.BT) {
        const float4 st = p.stats[row];
        rc.c = st.x + log2s;
        rc.lse2 = st.w;
        rc.f = fmaf(rc.zl2, st.w, 1.0f);
        rc.y = __float_as_int(st.y);
        rc.coef = scale * st.z;
      }
    } else {
      if (p.bias != nullptr && row < p.V) rc.bias2 = __ldg(p.bias + row) * kLog2e;
      rc.c = rc.bias2 + log2s;
      rc.y = row;
    }
    float gbias = 0.f;
    // kOwn > 1: the running sums of the other owner-class slots; before this pair's t-th block,
    // on_lsum / on_tsum / gbias hold slot t mod n_slots and the k-th of these slot (t + k) mod n_slots
    float cl_l1 = 0.f, cl_l2 = 0.f, cl_l3 = 0.f, cl_t1 = 0.f, cl_t2 = 0.f, cl_t3 = 0.f;
    float cl_g1 = 0.f, cl_g2 = 0.f, cl_g3 = 0.f;
    bool ok = true;
    // this CTA's writes into each slot, in content order (both halves: with an odd number of slots a slot
    // holds contents of either half), that had to wait for the slot's previous content to be consumed
    int waited[kSlots] = {};
    if (filt) {
      // O starts at zero (GEMM2 then always accumulates, whichever halves are skipped): this warp's 32
      // lanes of its 128 of the 256 accumulator columns
      for (int c = 0; c < 4; ++c)
        tmem_st_32cols_zero(tmem + (static_cast<uint32_t>(qq * 32) << 16) + kTmemO + static_cast<uint32_t>(hh * 128 + 32 * c));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sm.o_zero), lead_rank));
    }
    int u = 0;
    for (int j = pr; j < nt && ok; j += P, ++u) {
      if (kOwn > 1 && j > pr) {
        if constexpr (n_slots == 4) {
          float t = on_lsum;
          on_lsum = cl_l1, cl_l1 = cl_l2, cl_l2 = cl_l3, cl_l3 = t;
          t = on_tsum;
          on_tsum = cl_t1, cl_t1 = cl_t2, cl_t2 = cl_t3, cl_t3 = t;
          t = gbias;
          gbias = cl_g1, cl_g1 = cl_g2, cl_g2 = cl_g3, cl_g3 = t;
        } else {
          float t = on_lsum;
          on_lsum = cl_l1, cl_l1 = t;
          t = on_tsum;
          on_tsum = cl_t1, cl_t1 = t;
          t = gbias;
          gbias = cl_g1, cl_g1 = t;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full, u & 1, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(qq * 32) << 16) + kTmemS + static_cast<uint32_t>(hh * 128);
      // grad_W pass: the statistics of this half's 128 token columns (staged in the slot, and in global memory)
      if (kVocabRows && !__all_sync(0xffffffffu, mbar_wait(&sm.st_full, u & 1, abort))) {
        ok = false;
        break;
      }
      const typename Smem::Cfg::Stat* tstats = sm.colstats + (kVocabRows ? hh * 128 : 0);
      const float4* gst = kVocabRows ? p.stats + static_cast<size_t>(jb + j) * kPN + hh * 128 : nullptr;
      const int col0 = (jb + j) * kPN + hh * 128;
      // dS of this row's 128 columns in two chunks of 64, packed to bf16 pairs
      uint32_t pk0[32], pk1[32];
      {
        uint32_t ra[64], rb[64];
        tmem_ld_32cols(taddr, *reinterpret_cast<uint32_t(*)[32]>(&ra[0]));
        tmem_ld_32cols(taddr + 32u, *reinterpret_cast<uint32_t(*)[32]>(&ra[32]));
        tmem_ld_32cols(taddr + 64u, *reinterpret_cast<uint32_t(*)[32]>(&rb[0]));
        tmem_ld_32cols(taddr + 96u, *reinterpret_cast<uint32_t(*)[32]>(&rb[32]));
        tmem_wait_ld();
        // the logits tile is no longer needed: the next GEMM1 may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(s_empty_c);
        if (kOnline && !on_have_ref) {
          if (pr == 0 && j == 0 && hh == 0) {
            // the row's reference: its largest logit (+ bias) among the first 128 columns of block 0, in log2
            // units (the same number in every pair, so their accumulators share one scale)
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              m = fmaxf(m, fmaf(__uint_as_float(ra[i]), kLog2e, __ldg(p.colb2 + col0 + i)));
              m = fmaxf(m, fmaf(__uint_as_float(rb[i]), kLog2e, __ldg(p.colb2 + col0 + 64 + i)));
            }
            *on_mref = m;
            __syncwarp();
            if (lane == 0)
              for (int pp = 0; pp < P; ++pp)
                mbar_arrive_cluster(mapa_shared(smem_u32(&sm.mref_ready), static_cast<uint32_t>(2 * pp) + q));
          }
          if (!__all_sync(0xffffffffu, mbar_wait_cluster(&sm.mref_ready, 0, abort))) {
            ok = false;
            break;
          }
          on_ref = __ldcg(on_mref);
          on_have_ref = true;
        }
        // with the filter: is every entry of this row's half small, |dS| <= eps |w| with w the entry's
        // gradient weight (the row's for grad_input, the token column's for grad_W), i.e. the unscaled
        // p f - onehot below eps?  (fp32, before rounding; zero-weight entries are zero and count as small)
        bool small = true;
        int over = 0;
        const float fge = (kVocabRows && filt) ? p.filter_eps * fabsf(scale) : 0.f;
        int* const fov = (kVocabRows && filt) ? &over : nullptr;
        if (kOnline)
          online_chunk64(ra, col0, -on_ref, p.bias == nullptr && col0 + 64 <= p.V, p.colb2, p.bias, rc.y, on_lsum, on_zy,
                         on_ent, on_tsum);
        else
          ds_chunk64<kVocabRows>(ra, col0, rc, general, p.bias == nullptr && col0 + 64 <= p.V, p.colb2, tstats, gst,
                                 gbias, fge, fov);
        if (!kVocabRows && filt) small = filter_small_row(ra, rc, p.filter_eps);
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) pk0[i2] = pack_bf16x2(__uint_as_float(ra[2 * i2]), __uint_as_float(ra[2 * i2 + 1]));
        if (kOnline)
          online_chunk64(rb, col0 + 64, -on_ref, p.bias == nullptr && col0 + 128 <= p.V, p.colb2, p.bias, rc.y,
                         on_lsum, on_zy, on_ent, on_tsum);
        else
          ds_chunk64<kVocabRows>(rb, col0 + 64, rc, general, p.bias == nullptr && col0 + 128 <= p.V, p.colb2,
                                 tstats + 64, kVocabRows ? gst + 64 : nullptr, gbias, fge, fov);
        if (!kVocabRows && filt) small = filter_small_row(rb, rc, p.filter_eps) && small;
        if (kVocabRows && filt) small = (over == 0);
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) pk1[i2] = pack_bf16x2(__uint_as_float(rb[2 * i2]), __uint_as_float(rb[2 * i2 + 1]));
        if (kVocabRows) {
          // the statistics slot is free for the producer's next owned block
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.st_empty);
        }
        if (filt) {
          // this warp's verdict on its 32 rows of half hh of block j, published at once to every CTA of the
          // cluster: their producers and MMA threads skip the half when all 8 owner warps say "small"
          const bool all_small = __all_sync(0xffffffffu, small);
          if (lane == 0) {
            const int r = j % kFlagRing;
            const int slot = 4 * static_cast<int>(q) + qq;
            for (int c = 0; c < 2 * P; ++c) {
              st_shared_cluster_u32(mapa_shared(smem_u32(&sm.skipf[r][hh][slot]), static_cast<uint32_t>(c)),
                                    all_small ? 1u : 0u);
              mbar_arrive_cluster(mapa_shared(smem_u32(&sm.flag_full[r][hh]), static_cast<uint32_t>(c)));
            }
          }
        }
      }
      // content 2j + hh goes to slot (2j + hh) mod kSlots.  Unless it is the slot's first content, each pair
      // must be done with the slot's previous content before this content overwrites that pair's copy:
      // ds_free[slot][pp] completes when pair pp is (phase = this CTA's earlier writes into the slot that
      // waited).  A wait that gives up skips the writes; the warp leaves the loop after the send below.
      const int n_ds = 2 * j + hh;
      const int slot = n_ds % kSlots;
      const bool must_wait = n_ds >= kSlots;
      const uint32_t fpar = static_cast<uint32_t>(waited[slot]) & 1u;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2)
        if (2 * j + h2 >= kSlots) ++waited[(2 * j + h2) % kSlots];
      const bool own_free = __all_sync(0xffffffffu, !must_wait || mbar_wait_cluster(&sm.ds_free[slot][pr], fpar, abort));
      ok = ok && own_free;
      if (own_free) {
        uint8_t* const ds_row = sm.ds[slot] + static_cast<uint32_t>(rl) * 128u;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(ds_row + ((ch ^ (rl & 7)) << 4)) =
              make_uint4(pk0[4 * ch + 0], pk0[4 * ch + 1], pk0[4 * ch + 2], pk0[4 * ch + 3]);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(ds_row + kBox + ((ch ^ (rl & 7)) << 4)) =
              make_uint4(pk1[4 * ch + 0], pk1[4 * ch + 1], pk1[4 * ch + 2], pk1[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      // with the filter, a half every pair skips is not sent: the other pairs' receivers get its byte count
      // as a bare transaction completion (after the slot wait above, so blocks still complete in order).
      // A verdict wait that gave up sends the data (the kernel is winding down by then).
      bool send = true;
      if (filt && lane == 0) send = filter_verdict(sm, j, hh, abort) != 1;
      // the warp's 32 rows are two contiguous 4 KB runs (one per 64-column box); each lane moves 16-byte
      // pieces of them, so that every store instruction writes 512 consecutive bytes of the peer's slot
      send = __shfl_sync(0xffffffffu, send, 0);
      const uint8_t* const src = sm.ds[slot] + static_cast<uint32_t>(qq) * 4096u;
      for (int pp = 0; pp < P && ok; ++pp) {
        if (pp == pr) continue;
        const uint32_t dst_rank = static_cast<uint32_t>(2 * pp) + q;
        const uint32_t bar = mapa_shared(smem_u32(&sm.rx_full[slot]), dst_rank);
        if (must_wait && !__all_sync(0xffffffffu, mbar_wait_cluster(&sm.ds_free[slot][pp], fpar, abort))) {
          ok = false;
          break;
        }
        if (send) {
          const uint32_t dst = mapa_shared(smem_u32(src), dst_rank);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t off = static_cast<uint32_t>(i >> 3) * kBox + static_cast<uint32_t>(i & 7) * 512u +
                                 static_cast<uint32_t>(lane) * 16u;
            st_async_v4(dst + off, *reinterpret_cast<const uint4*>(src + off), bar);
          }
        } else if (lane == 0) {
          mbar_complete_tx_cluster(bar, 2u * 4096u);
        }
      }
      // (every lane takes the same exit)
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // this warp's rows of the slot are written here and on their way to the other pairs: one of the 8
      // arrivals the MMA issuer waits for (no barrier between the epilogue warps, so none can be left
      // waiting for a warp that gave up)
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sm.ds_full[slot]), lead_rank));
    }

    // online form: every pair's partial sums of this row combined into the row's outputs (online_row_finish),
    // or, in a vocabulary-split unit, into the unit's partial statistics
    float on_c1 = 0.f, on_c2 = 0.f;
    bool on_row_ok = true;
    if (kOnline) {
      if (ok && !on_have_ref) {
        // a pair that owned no block still needs the reference
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&sm.mref_ready, 0, abort))) {
          ok = false;
        } else {
          on_ref = __ldcg(on_mref);
          on_have_ref = true;
        }
      }
      if (ok) {
        if (kOwn > 1) {
          // (the target logit is a maximum: any class may carry it)
          for (int sl = 0; sl < n_slots; ++sl)
            on_part[(pr + sl * P) * 2 + hh] = make_float4(slot_sum(on_lsum, cl_l1, cl_l2, cl_l3, sl, u, n_slots), on_zy,
                                                          slot_sum(on_tsum, cl_t1, cl_t2, cl_t3, sl, u, n_slots), 0.f);
        } else {
          on_part[pr * 2 + hh] = make_float4(on_lsum, on_zy, on_tsum, 0.f);
        }
        __syncwarp();
        if (lane == 0)
          for (int pp = 0; pp < P; ++pp)
            mbar_arrive_cluster(mapa_shared(smem_u32(&sm.part_ready), static_cast<uint32_t>(2 * pp) + q));
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&sm.part_ready, 0, abort))) ok = false;
      }
      if (ok) {
        float L = 0.f, zy = -INFINITY, T = 0.f;
        for (int pp = 0; pp < (kOwn > 1 ? kMaxPairs : P); ++pp)
          for (int h2 = 0; h2 < 2; ++h2) {
            const float4 v = __ldcg(on_part + pp * 2 + h2);
            L += v.x;
            zy = fmaxf(zy, v.y);
            T += v.z;
          }
        if (su >= 0) {
          if (pr == 0 && hh == 0) p.vs_stat[static_cast<size_t>(su) * 256 + rloc] = make_float4(L, zy, T, on_ref);
        } else {
          const OnlineRow fr = online_row_finish(p, row, on_ref, L, zy, T, rc.y, on_u, scale, pr == 0 && hh == 0);
          on_c1 = fr.c1;
          on_c2 = fr.c2;
          on_row_ok = fr.ok;
        }
      }
    }

    const bool o_ready = ok && __all_sync(0xffffffffu, mbar_wait(&sm.o_full, 0, abort));
    if (o_ready && kVocabRows && su < 0) {
      // grad_W rows: this warp's 32 rows x the 128 columns of half hh, staged in the operand stages and dS
      // slots (free: every MMA of the pair has completed, every dS sent here has been consumed, and the
      // producer issues nothing more in this unit), then one bulk copy per row, a bulk reduce-add when
      // accumulating (old + new, as the register path adds them); the copies have read the stage before
      // the cluster barrier after which the grad_bias gather reuses it
      tc_fence_after();
      const int n_chunks = (hc + 31) / 32;
      uint8_t* const my_row = &sm.stage[0][0] + (static_cast<size_t>(warp) * 32 + lane) * kDrainRowBytes;
      for (int c = 4 * hh; c < 4 * hh + 4 && c < n_chunks; ++c) {
        uint32_t vv[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(qq * 32) << 16) + kTmemO + 32u * c, vv);
        tmem_wait_ld();
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)
          *reinterpret_cast<uint4*>(my_row + (c - 4 * hh) * 128 + 16 * g4) =
              make_uint4(vv[4 * g4], vv[4 * g4 + 1], vv[4 * g4 + 2], vv[4 * g4 + 3]);
      }
      const int ncols = min(128, hc - 128 * hh);   // this half's columns inside H (a multiple of 8)
      if (row < p.V && p.grad_W != nullptr && ncols > 0) {
        fence_proxy_async_smem();
        const int orow = p.row_perm != nullptr ? p.row_perm[row] : row;
        float* const out = p.grad_W + static_cast<size_t>(orow) * p.H + h0 + 128 * hh;
        if (p.accumulate)
          bulk_add_f32_1d(out, my_row, 4u * static_cast<uint32_t>(ncols));
        else
          bulk_store_1d(out, my_row, 4u * static_cast<uint32_t>(ncols));
        bulk_commit_wait_read();
      }
    } else if (o_ready) {
      tc_fence_after();
      const int n_chunks = (hc + 31) / 32;
      for (int c = hh; c < n_chunks; c += 2) {
        uint32_t vv[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(qq * 32) << 16) + kTmemO + 32u * c, vv);
        tmem_wait_ld();
        const int cb = 32 * c;
        if (su >= 0) {
          // split unit: the raw accumulator columns of this pair, for the merge kernel (grad_W pass: not
          // needed when only grad_bias is asked for)
          if (kVocabRows && p.grad_W == nullptr) continue;
          float* out = p.vs_o + (static_cast<size_t>(su) * 256 + rloc) * (P * kHc) + pr * kHc + cb;
#pragma unroll
          for (int g4 = 0; g4 < 8; ++g4)
            if (cb + 4 * g4 + 4 <= hc)
              *reinterpret_cast<float4*>(out + 4 * g4) =
                  make_float4(__uint_as_float(vv[4 * g4 + 0]), __uint_as_float(vv[4 * g4 + 1]),
                              __uint_as_float(vv[4 * g4 + 2]), __uint_as_float(vv[4 * g4 + 3]));
        } else if (!kVocabRows) {
          // (online: a row outside the safe range is left to the classic pass; classic behind an online
          // pass: only such rows)
          const bool write_row = kOnline ? on_row_ok : (p.row_redo == nullptr || (row < p.BT && p.row_redo[row] != 0u));
          if (row < p.BT && write_row) {
            uint16_t* out = p.grad_input + static_cast<size_t>(row) * p.H + h0 + cb;
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              if (cb + 8 * g8 + 8 <= hc) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(vv[8 * g8 + e]);
                if (kOnline) {
                  float wy[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                  if (on_c2 != 0.f) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(p.Wmat + static_cast<size_t>(rc.y) * p.H + h0 + cb +
                                                                     8 * g8);
                    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      wy[2 * e] = bf16_lo(ww[e]);
                      wy[2 * e + 1] = bf16_hi(ww[e]);
                    }
                  }
#pragma unroll
                  for (int e = 0; e < 8; ++e) o[e] = fmaf(on_c1, o[e], on_c2 * wy[e]);
                }
                if (p.accumulate) {
                  const uint4 old = *reinterpret_cast<const uint4*>(out + 8 * g8);
                  const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    o[2 * e] += bf16_lo(ow[e]);
                    o[2 * e + 1] += bf16_hi(ow[e]);
                  }
                }
                *reinterpret_cast<uint4*>(out + 8 * g8) = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                                                     pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
              }
            }
          }
        } else {
          if (row < p.V && p.grad_W != nullptr) {
            const int orow = p.row_perm != nullptr ? p.row_perm[row] : row;
            float* out = p.grad_W + static_cast<size_t>(orow) * p.H + h0 + cb;
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
              if (cb + 4 * g4 + 4 <= hc) {
                float4 o = make_float4(__uint_as_float(vv[4 * g4 + 0]), __uint_as_float(vv[4 * g4 + 1]),
                                       __uint_as_float(vv[4 * g4 + 2]), __uint_as_float(vv[4 * g4 + 3]));
                if (p.accumulate) {
                  const float4 old = *reinterpret_cast<const float4*>(out + 4 * g4);
                  o.x += old.x;
                  o.y += old.y;
                  o.z += old.z;
                  o.w += old.w;
                }
                *reinterpret_cast<float4*>(out + 4 * g4) = o;
              }
            }
          }
        }
      }
    }
    gbias_out = kOwn > 1 ? slot_sum(gbias, cl_g1, cl_g2, cl_g3, 0, u, n_slots) : gbias;
    if (kOwn > 1) {
      gbias_c1 = slot_sum(gbias, cl_g1, cl_g2, cl_g3, 1, u, n_slots);
      gbias_c2 = slot_sum(gbias, cl_g1, cl_g2, cl_g3, 2, u, n_slots);
      gbias_c3 = slot_sum(gbias, cl_g1, cl_g2, cl_g3, 3, u, n_slots);
    }
  }

  tc_fence_before();
  cluster_sync();
  // grad_W pass: every MMA of the cluster has completed by now (each MMA thread waited for its drain, each
  // epilogue for o_full, before the barrier), so the dS blocks are free and gather the grad_bias partials:
  // [pair][half][row] in pair 0's CTA with the same rows, added there in pair and half order
  float* const gb_gather = reinterpret_cast<float*>(&sm.ds[0][0]);
  if (kVocabRows) {
    if (warp < kEpiWarps) {
      const int rl = (warp & 3) * 32 + lane;
      st_shared_cluster_f32(mapa_shared(smem_u32(gb_gather + (pr * 2 + (warp >> 2)) * kTileM + rl), q), gbias_out);
      if (kOwn > 1) {
        // the other slots' classes: pr + s P
        const float gs[3] = {gbias_c1, gbias_c2, gbias_c3};
#pragma unroll
        for (int sl = 1; sl < 4; ++sl)
          if (sl < n_slots)
            st_shared_cluster_f32(mapa_shared(smem_u32(gb_gather + ((pr + sl * P) * 2 + (warp >> 2)) * kTileM + rl), q),
                                  gs[sl - 1]);
      }
    }
    cluster_sync();
  }
  if (kVocabRows && pr == 0 && warp < 4 && hgroup == 0 && p.grad_bias != nullptr && !sm.abort) {
    const int rl = warp * 32 + lane;
    const int row = r0 + rl;
    if (row < p.V) {
      float acc = 0.f;
      for (int pp = 0; pp < (kOwn > 1 ? kMaxPairs : P); ++pp)
        acc += gb_gather[(pp * 2) * kTileM + rl] + gb_gather[(pp * 2 + 1) * kTileM + rl];
      if (su >= 0) {
        p.vs_gb[static_cast<size_t>(su) * 256 + static_cast<int>(q) * kTileM + rl] = acc;   // for dw_vmerge_kernel
      } else {
        const int orow = p.row_perm != nullptr ? p.row_perm[row] : row;
        p.grad_bias[orow] = p.accumulate ? p.grad_bias[orow] + acc : acc;
      }
    }
  }
  if (kTmem == kTmemOneUnit && warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort) atomicOr(status, kStatusTimeout);
}

// Work units of a gradient pass, in launch order: n_whole clusters over all column blocks (row pair
// u / groups, H group u % groups), then for the last row pairs, from rp_tail0 on, groups x nsplit clusters,
// each over one of nsplit consecutive ranges of the nt column blocks (split units, numbered
// su = (tail row pair x groups + group) x nsplit + part), which a merge kernel combines (online_vmerge_kernel
// for the online grad_input pass, dw_vmerge_kernel for the grad_W pass).  Splitting the row pairs of a
// partly filled last wave shortens that wave.
// Uneven form (jsplit > 0, nsplit = 2): each of the n_tail split row-pair clusters has a large part over
// blocks [0, jsplit) and a small part over [jsplit, nt); all large parts are launched first, so that the
// free slots of the last wave take the small parts (n_tail / (slots - n_tail) of them each).
struct UnitPlan {
  int groups, n_whole, rp_tail0, nsplit, nt;
  int jsplit, n_tail;
};
struct Unit {
  int row_pair, hgroup, jb, je, su;
};
__device__ __forceinline__ Unit unit_of(const UnitPlan& plan, int c) {
  Unit u{c / plan.groups, c % plan.groups, 0, plan.nt, -1};
  if (c >= plan.n_whole) {
    const int k = c - plan.n_whole;
    int part, ug;
    if (plan.jsplit > 0) {
      part = k / plan.n_tail;
      ug = k % plan.n_tail;
      u.jb = part == 0 ? 0 : plan.jsplit;
      u.je = part == 0 ? plan.jsplit : plan.nt;
    } else {
      part = k % plan.nsplit;
      ug = k / plan.nsplit;
      u.jb = (part * plan.nt) / plan.nsplit;
      u.je = ((part + 1) * plan.nt) / plan.nsplit;
    }
    u.su = ug * plan.nsplit + part;
    u.row_pair = plan.rp_tail0 + ug / plan.groups;
    u.hgroup = ug % plan.groups;
  }
  return u;
}

// A CTA's gradient work: TMEM allocated once, then the one unit `fixed` (kQueue false), or (kQueue) the
// units it claims from the work queue, CTA 0 of the cluster claiming and handing the index to every CTA
// (claim_next: the first before any unit, each next one during the unit before it), until none is left.
// The barriers are initialised again for every unit: dgrad_pair_body ends with every arrival on them
// consumed or ordered before its last cluster barrier, which also orders the next claim before every
// CTA reads it.  A unit that gave up on a wait stops the cluster.  (A template flag rather than a run-time
// one, so that the one-unit kernels keep their register allocation.)
template <bool kVocabRows, bool kFilter, bool kOnline, int kSlots, int kOwn, bool kQueue>
__device__ __forceinline__ void run_units(const CUtensorMap& tm_rows, const CUtensorMap& tm_cols, const PairParams& p,
                                          uint32_t* __restrict__ status, const Unit& fixed, const UnitPlan& plan,
                                          const WorkQueue& wq) {
  // the classic passes behind an online grad_input pass run only when it asked for them
  if (p.gate != nullptr && *reinterpret_cast<const volatile uint32_t*>(p.gate) == 0u) return;
  auto* const smp = pair_smem_of<kVocabRows, kFilter, kSlots>();
  if (smp == nullptr) {
    if (threadIdx.x == 0) atomicOr(status, kStatusInternal);
    return;
  }
  if constexpr (!kQueue) {
    // (the body allocates and frees TMEM itself)
    dgrad_pair_body<kVocabRows, kFilter, kOnline, kSlots, kOwn, kTmemOneUnit>(
        tm_rows, tm_cols, p, status, fixed.row_pair, fixed.hgroup, fixed.jb, fixed.je, fixed.su, wq);
  } else {
    auto& sm = *smp;
    if ((threadIdx.x >> 5) == kMmaWarp) {
      tmem_alloc_pair(&sm.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    }
    // the launch behind this one (side behind main, single-pair behind side) may start on the SMs left free
    griddep_launch_dependents();
    uint32_t* const counts = wq.role == kRoleSide ? wq.side_count : wq.role == kRoleSingle ? wq.single_count : nullptr;
    if (blockIdx.x == 0 && threadIdx.x == 0 && counts != nullptr) atomicAdd(counts, 1u);
    const uint32_t rank = cluster_ctarank();
    const int n_sub = wq.role == kRoleSingle ? wq.side_chunks : 1;
    if (rank == 0 && threadIdx.x == 0) {
      sm.q_sub = 0;
      sm.q_took = 0;
    }
    // The grad_W pass (units of BT / 256 blocks: short ones at small BT) claims each next unit inside the
    // unit before it, while the accumulator drains (claim_next in dgrad_pair_body): 2.70 -> 2.64 ms for
    // qwen3's pass of 16-block units.  The grad_input pass claims between its units, behind one more
    // cluster barrier: its units are long, and with the claim inside its body, or the claim's code shared
    // with the grad_W pass, its kernel compiled to one that took 0.1-0.2 ms longer at the long workload.
    if constexpr (kVocabRows) {
      if (rank == 0 && threadIdx.x == 0) claim_next(sm, wq, status, 2 * p.P, false);
      cluster_sync();
      for (;;) {
        // (the unit's claim: written by CTA 0 before the cluster barrier above, or before the previous
        // unit's last one; the next claim is written only after this unit's first cluster barrier)
        const int v = *reinterpret_cast<volatile int*>(&sm.claim);
        if (v < 0) break;
        const int c = v / n_sub;
        const Unit u = wq.role == kRoleMain ? Unit{c / wq.main_groups, c % wq.main_groups, 0, plan.nt, -1}
                                            : Unit{wq.row_pairs - 1 - c / wq.side_groups,
                                                   (c % wq.side_groups) * n_sub + v % n_sub, 0, plan.nt, -1};
        // (the body ends with a cluster barrier after every access of the unit's barriers, TMEM and
        // shared memory by the other CTAs, so the next unit may initialise them at once)
        dgrad_pair_body<kVocabRows, kFilter, kOnline, kSlots, kOwn, kTmemHeld>(
            tm_rows, tm_cols, p, status, u.row_pair, u.hgroup, u.jb, u.je, u.su, wq);
      }
    } else {
      for (;;) {
        if (rank == 0 && threadIdx.x == 0) {
          const int sub = sm.q_sub;
          if (sub == 0) {
            int cl = (*reinterpret_cast<volatile uint32_t*>(status) & kStatusTimeout) != 0u ? -1 : claim_unit(wq);
            if (cl == -2) {
              atomicOr(status, kStatusInternal);
              cl = -1;
            }
            if (cl >= 0 && !sm.q_took && counts != nullptr) atomicAdd(counts + 1, 1u);
            if (cl >= 0 && wq.role == kRoleSingle && wq.single_units != nullptr) atomicAdd(wq.single_units, 1u);
            if (cl >= 0) sm.q_took = 1;
            sm.q_unit = cl;
          }
          sm.q_sub = sub + 1 == n_sub ? 0 : sub + 1;
          const int v = sm.q_unit < 0 ? -1 : sm.q_unit * n_sub + sub;
          for (int r = 0; r < 2 * p.P; ++r)
            st_shared_cluster_u32(mapa_shared(smem_u32(&sm.claim), static_cast<uint32_t>(r)), static_cast<uint32_t>(v));
        }
        cluster_sync();
        const int v = *reinterpret_cast<volatile int*>(&sm.claim);
        if (v < 0) break;
        const int c = v / n_sub;
        const Unit u = wq.role == kRoleMain ? Unit{c / wq.main_groups, c % wq.main_groups, 0, plan.nt, -1}
                                            : Unit{wq.row_pairs - 1 - c / wq.side_groups,
                                                   (c % wq.side_groups) * n_sub + v % n_sub, 0, plan.nt, -1};
        dgrad_pair_body<kVocabRows, kFilter, kOnline, kSlots, kOwn, kTmemHeld>(
            tm_rows, tm_cols, p, status, u.row_pair, u.hgroup, u.jb, u.je, u.su, wq);
        // every CTA is done with the unit (and has read sm.claim) before the next claim is handed out
        cluster_sync();
      }
    }
    // a side grid completes only after the main grid beside it, a single-pair grid only after the side grid
    // (and so the main grid), so that what follows on the stream sees all of them
    if (wq.role != kRoleMain) griddep_wait_primary();
    // (every CTA of the cluster has passed a cluster barrier after its last TMEM access)
    if ((threadIdx.x >> 5) == kMmaWarp) {
      tc_fence_after();
      tmem_dealloc_pair(sm.tmem_base, kTmemCols);
    }
  }
}

// One gradient pass: without a queue, cluster blockIdx.x / 2P is work unit unit_of(plan, .); with one
// (kQueue), a persistent cluster of the main, side or single-pair launch (WorkQueue; the side launch's
// pairs with kOwn = 2, the single-pair launch's with kOwn = 4).
template <bool kVocabRows, bool kFilter, int kSlots, int kOwn = 1, bool kQueue = false>
__global__ void __launch_bounds__(kThreads, 1)
dgrad_pair_kernel(const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_cols,
                  const PairParams p, uint32_t* __restrict__ status, const UnitPlan plan, const WorkQueue wq) {
  const Unit u = unit_of(plan, static_cast<int>(blockIdx.x) / (2 * p.P));
  run_units<kVocabRows, kFilter, false, kSlots, kOwn, kQueue>(tm_rows, tm_cols, p, status, u, plan, wq);
}

// The grad_input pass without a prior LSE pass: the same cluster layout as dgrad_pair_kernel<false>.
template <int kSlots, int kOwn = 1, bool kQueue = false>
__global__ void __launch_bounds__(kThreads, 1)
dgrad_online_kernel(const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_cols,
                    const PairParams p, uint32_t* __restrict__ status, const UnitPlan plan, const WorkQueue wq) {
  const Unit u = unit_of(plan, static_cast<int>(blockIdx.x) / (2 * p.P));
  run_units<false, false, true, kSlots, kOwn, kQueue>(tm_rows, tm_cols, p, status, u, plan, wq);
}

// The vocabulary rows of token-split units of the grad_W pass: grad_W[row] = sum over parts, in order, of
// their partial rows (plus the old value when accumulating), the same for grad_bias.  One CTA of 128
// threads per row.
__global__ void __launch_bounds__(128) dw_vmerge_kernel(const PairParams p, const UnitPlan plan) {
  const int t = static_cast<int>(blockIdx.x) / 256, rloc = static_cast<int>(blockIdx.x) % 256;
  const int row = (plan.rp_tail0 + t) * 256 + rloc;
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.vs_count != nullptr)
    *p.vs_count = static_cast<uint32_t>(gridDim.x / 256 * plan.groups * plan.nsplit);
  if (row >= p.V) return;
  const int ns = plan.nsplit;
  const int orow = p.row_perm != nullptr ? p.row_perm[row] : row;
  const int span = p.P * kHc;
  if (p.grad_W != nullptr) {
    for (int h = 4 * static_cast<int>(threadIdx.x); h < p.H; h += 4 * 128) {
      const int g = h / span, col = h - g * span;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int v = 0; v < ns; ++v) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(
            p.vs_o + (static_cast<size_t>((t * plan.groups + g) * ns + v) * 256 + rloc) * span + col));
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
      float4* out = reinterpret_cast<float4*>(p.grad_W + static_cast<size_t>(orow) * p.H + h);
      if (p.accumulate) {
        const float4 old = *out;
        acc.x += old.x;
        acc.y += old.y;
        acc.z += old.z;
        acc.w += old.w;
      }
      *out = acc;
    }
  }
  if (threadIdx.x == 0 && p.grad_bias != nullptr) {
    float acc = 0.f;
    // (group 0's units carry grad_bias)
    for (int v = 0; v < ns; ++v) acc += __ldcg(p.vs_gb + static_cast<size_t>(t * plan.groups * ns + v) * 256 + rloc);
    p.grad_bias[orow] = p.accumulate ? p.grad_bias[orow] + acc : acc;
  }
}

constexpr int kMaxSplitParts = 16;

// The rows of vocabulary-split units: per row, the units' partial sums rescaled to the largest of their
// references R and added (L = sum_v 2^(ref_v - R) L_v, the same for T; z_y from the unit that saw the
// target), then the row's outputs as in the pass itself (online_row_finish) and
// grad_input[row] = c1 sum_v 2^(ref_v - R) O_v[row] + c2 W[y].  One CTA of 128 threads per row.
__global__ void __launch_bounds__(128) online_vmerge_kernel(const PairParams p, const UnitPlan plan) {
  const int t = static_cast<int>(blockIdx.x) / 256, rloc = static_cast<int>(blockIdx.x) % 256;
  const int row = (plan.rp_tail0 + t) * 256 + rloc;
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.vs_count != nullptr)
    *p.vs_count = static_cast<uint32_t>(gridDim.x / 256 * plan.groups * plan.nsplit);
  if (row >= p.BT) return;
  const int ns = plan.nsplit;
  float ref[kMaxSplitParts], w[kMaxSplitParts];
  float R = -INFINITY;
#pragma unroll
  for (int v = 0; v < kMaxSplitParts; ++v) {
    ref[v] = -INFINITY;
    if (v < ns) {
      // (group 0's units: every group sees the same logits)
      ref[v] = __ldcg(&p.vs_stat[static_cast<size_t>(t * plan.groups * ns + v) * 256 + rloc].w);
      R = fmaxf(R, ref[v]);
    }
  }
  float L = 0.f, zy = -INFINITY, T = 0.f;
  bool fin = true;
#pragma unroll
  for (int v = 0; v < kMaxSplitParts; ++v) {
    w[v] = 0.f;
    if (v < ns) {
      const float4 st = __ldcg(&p.vs_stat[static_cast<size_t>(t * plan.groups * ns + v) * 256 + rloc]);
      w[v] = ex2_approx(ref[v] - R);
      L = fmaf(st.x, w[v], L);
      T = fmaf(st.z, w[v], T);
      zy = fmaxf(zy, st.y);
      fin = fin && st.x < 0x1p115f;   // each part's accumulator stayed in the safe range
    }
  }
  if (!fin) L = INFINITY;
  const int64_t yy = p.target[row];
  const int y = (yy != p.ignore_index && yy >= 0 && yy < p.V) ? static_cast<int>(yy) : -1;
  const float u = p.grad_tok != nullptr ? p.grad_tok[row] : 1.0f;
  const OnlineRow fr = online_row_finish(p, row, R, L, zy, T, y, u, *p.scale, threadIdx.x == 0);
  if (!fr.ok) return;
  const int span = p.P * kHc;   // columns of one unit
  for (int h = 8 * static_cast<int>(threadIdx.x); h < p.H; h += 8 * 128) {
    const int g = h / span, col = h - g * span;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int v = 0; v < kMaxSplitParts; ++v) {
      if (v < ns) {
        const float* src = p.vs_o + (static_cast<size_t>((t * plan.groups + g) * ns + v) * 256 + rloc) * span + col;
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src + 4));
        o[0] = fmaf(w[v], a.x, o[0]);
        o[1] = fmaf(w[v], a.y, o[1]);
        o[2] = fmaf(w[v], a.z, o[2]);
        o[3] = fmaf(w[v], a.w, o[3]);
        o[4] = fmaf(w[v], b.x, o[4]);
        o[5] = fmaf(w[v], b.y, o[5]);
        o[6] = fmaf(w[v], b.z, o[6]);
        o[7] = fmaf(w[v], b.w, o[7]);
      }
    }
    float wy[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (fr.c2 != 0.f) {
      const uint4 wv = *reinterpret_cast<const uint4*>(p.Wmat + static_cast<size_t>(y) * p.H + h);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        wy[2 * e] = bf16_lo(ww[e]);
        wy[2 * e + 1] = bf16_hi(ww[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = fmaf(fr.c1, o[e], fr.c2 * wy[e]);
    uint16_t* out = p.grad_input + static_cast<size_t>(row) * p.H + h;
    if (p.accumulate) {
      const uint4 old = *reinterpret_cast<const uint4*>(out);
      const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[2 * e] += bf16_lo(ow[e]);
        o[2 * e + 1] += bf16_hi(ow[e]);
      }
    }
    *reinterpret_cast<uint4*>(out) =
        make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
  }
}

// Both gradient passes in one grid, so that the grad_W pass's clusters take the SMs the grad_input pass's
// last wave leaves idle: clusters 0 .. n_in-1 (in the grad_input pass's own order, row pairs fastest) run
// the grad_input pass, the rest the grad_W pass.  Both passes have the same number of pairs per cluster.
template <bool kFilter, int kSlots>
__global__ void __launch_bounds__(kThreads, 1)
dgrad_both_kernel(const __grid_constant__ CUtensorMap tm_hidden, const __grid_constant__ CUtensorMap tm_w,
                  const PairParams p_in, const PairParams p_w, uint32_t* __restrict__ status, int n_in,
                  int in_row_pairs, int w_row_pairs) {
  const int c = static_cast<int>(blockIdx.x) / (2 * p_in.P);
  const UnitPlan none{};
  const WorkQueue no_queue{};
  if (c < n_in) {
    const Unit u{c % in_row_pairs, c / in_row_pairs, 0, -1, -1};
    run_units<false, kFilter, false, kSlots, 1, false>(tm_hidden, tm_w, p_in, status, u, none, no_queue);
  } else {
    const int cw = c - n_in;
    const Unit u{cw % w_row_pairs, cw / w_row_pairs, 0, -1, -1};
    run_units<true, kFilter, false, kSlots, 1, false>(tm_w, tm_hidden, p_w, status, u, none, no_queue);
  }
}

// Four pairs per cluster (clusters of 8 CTAs, every logits tile computed once per pass when H is a
// multiple of 1024; four dS half-slots per CTA and three operand stages), for the exact passes whose
// units run over at least kFourPairsMinBlocks column blocks: the pipeline fill of 2P steps per unit costs
// too much on shorter units (a grad_W pass over 4096 tokens has 16 blocks per unit).  Measured at
// BT = 65535, H = 1024, V = 176245: 83.9 ms per step against 91.7 with two pairs.
constexpr int kFourPairsMinBlocks = 64;
// ... or at least this many when the pass runs persistent with side clusters (launch_corun), which take
// up what the fill costs the shorter units: qwen3's grad_W pass (16 blocks per unit) 2.75 ms with four
// pairs and side clusters against 2.85 with two pairs.
constexpr int kFourPairsMinBlocksSide = 16;
// dS half-slots per CTA with four pairs
constexpr int kFourPairSlots = 4;
// Persistent scheduling with side clusters (launch_corun) needs at least this many waves of main units.
constexpr int kCoRunMinWaves = 3;

// Pairs per cluster: 4 when allowed (see above) and the number of 256-wide H chunks divides by 4, else 2
// when it is even, else 3 when it divides by 3, else 1.
int pairs_per_cluster(int h_chunks, bool four_ok) {
  if (four_ok && h_chunks % 4 == 0) return 4;
  if (h_chunks % 2 == 0) return 2;
  if (h_chunks % 3 == 0) return 3;
  return 1;
}

// Kernel parameters of one pass; h_chunks receives the number of 256-wide H chunks it covers.
template <bool kVocabRows>
PairParams make_pair_params(const DgPairArgs& a, int* h_chunks) {
  PairParams p{};
  p.bias = a.bias;
  p.stats = a.stats;
  p.stats_ct = a.stats_ct;
  p.colb2 = a.colb2;
  p.scale = a.scale;
  p.zf_neg = a.zf_neg;
  p.z_loss = a.z_loss;
  p.accumulate = a.accumulate ? 1 : 0;
  p.filter_eps = a.filter_eps;
  p.skip_count = a.skip_count;
  p.row_perm = a.row_perm;
  p.debug_stall_us = a.debug_stall_us;
  p.BT = a.BT;
  p.V = a.V;
  p.H = a.H;
  p.n_rows = kVocabRows ? a.V : a.BT;
  p.n_cols = kVocabRows ? a.BT : a.V;
  p.num_kb = (a.H + kBK - 1) / kBK;
  p.grad_input = a.grad_input;
  p.grad_W = a.grad_W;
  p.grad_bias = a.grad_bias;
  p.gate = a.gate;
  p.target = a.target;
  p.ignore_index = a.ignore_index;
  p.grad_tok = a.grad_tok;
  p.Wmat = a.Wmat;
  p.mref_g = a.mref_g;
  p.part_g = a.part_g;
  p.entropy_out = a.entropy_out;
  p.row_redo = a.row_redo;
  p.stats_out = a.stats_out;
  p.stats_ct_out = a.stats_ct_out;
  p.row_loss = a.row_loss;
  p.loss_tok = a.loss_tok;
  p.zf_neg_out = a.zf_neg_out;
  p.fallback = a.fallback;
  // with only grad_bias requested one H chunk suffices (the GEMM2 result is not stored)
  *h_chunks = (kVocabRows && p.grad_W == nullptr) ? 1 : (p.H + kHc - 1) / kHc;
  const int n_blocks = (p.n_cols + kPN - 1) / kPN;
  p.P = pairs_per_cluster(*h_chunks, !(p.filter_eps > 0.f) && n_blocks >= kFourPairsMinBlocks);
  return p;
}

int row_pairs_of(const PairParams& p) { return (p.n_rows + 2 * kTileM - 1) / (2 * kTileM); }

// Whether a pass that make_pair_params gave two pairs (units of kFourPairsMinBlocksSide ..
// kFourPairsMinBlocks - 1 column blocks) takes four instead: when its H chunks divide by 4 and it will
// run persistent with side clusters (launch_corun's conditions; res4: resident 8-CTA clusters, 0 unknown).
bool four_pairs_with_side(const PairParams& p, int h_chunks, int splits_option, const DgPairArgs& a, int res4) {
  const int n_blocks = (p.n_cols + kPN - 1) / kPN;
  return p.P == 2 && h_chunks % 4 == 0 && !(p.filter_eps > 0.f) && a.work_q != nullptr && splits_option == 0 &&
         n_blocks >= kFourPairsMinBlocksSide && res4 > 0 &&
         row_pairs_of(p) * (h_chunks / 4) >= kCoRunMinWaves * res4;
}

cudaLaunchConfig_t cluster_config(dim3 grid, size_t smem, int P, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2 * P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of 2P CTAs of this kernel resident at once (-1 if the query fails).  While the stream is being
// captured into a CUDA graph the query is not made: 0, so that call plans no split tail and a later call
// asks again.
template <class Kernel>
int resident_clusters(Kernel kern, size_t smem, int P, cudaStream_t stream) {
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (capture != cudaStreamCaptureStatusNone) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t q = cluster_config(dim3(2 * P, 1, 1), smem, P, stream, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess) {
    (void)cudaGetLastError();
    n = -1;
  }
  return n;
}

// Split plan of a pass over row_pairs x groups clusters of nt column blocks (see UnitPlan).  forced: 0 =
// split the row pairs of a partly filled last wave of `slots` resident clusters, each into
// slots / (their clusters) parts; 1 = never; k >= 2 = every row pair into k parts.  Parts hold at least 4
// column blocks; at most kMaxSplitParts parts and su_cap split units.
//   With `uneven`, a last wave whose row pairs fill more than half of the slots (too many for equal
// parts) is split unevenly instead: each of its n_tail clusters into a part of jsplit blocks and the
// rest, so that the slots - n_tail free slots take the rests side by side and finish with the large parts.
UnitPlan make_plan(int row_pairs, int groups, int nt, int slots, int forced, int su_cap, bool uneven) {
  UnitPlan plan{groups, row_pairs * groups, row_pairs, 1, nt, 0, 0};
  const int units = row_pairs * groups;
  int tail_rp = 0, nsplit = 1;
  if (forced >= 2) {
    tail_rp = row_pairs;
    nsplit = forced;
  } else if (forced == 0 && slots > 0 && units % slots != 0) {
    tail_rp = std::min(row_pairs, (units % slots + groups - 1) / groups);
    nsplit = slots / (tail_rp * groups);
  }
  if (tail_rp > 0) nsplit = std::min({nsplit, kMaxSplitParts, nt / 4, su_cap / (tail_rp * groups)});
  if (tail_rp > 0 && nsplit < 2 && uneven && forced == 0 && tail_rp * groups < slots) {
    // m small parts run back to back on each free slot; a split cluster also costs a fixed ~7 block steps
    // (measured ~30 us at H = 1024: pipeline fill, reference, partial write-out), so the split point
    // balances jsplit + c against m (nt - jsplit + c): jsplit = (m nt + (m - 1) c) / (m + 1)
    constexpr int kPartCostBlocks = 7;
    const int n_tail = tail_rp * groups;
    const int m = (n_tail + (slots - n_tail) - 1) / (slots - n_tail);
    const int jsplit = (m * nt + (m - 1) * kPartCostBlocks) / (m + 1);
    if (2 * n_tail <= su_cap && jsplit >= 4 && nt - jsplit >= 4) {
      plan.nsplit = 2;
      plan.jsplit = jsplit;
      plan.n_tail = n_tail;
      plan.rp_tail0 = row_pairs - tail_rp;
      plan.n_whole = plan.rp_tail0 * groups;
    }
    return plan;
  }
  if (tail_rp == 0 || nsplit < 2) return plan;
  plan.nsplit = nsplit;
  plan.n_tail = tail_rp * groups;
  plan.rp_tail0 = row_pairs - tail_rp;
  plan.n_whole = plan.rp_tail0 * groups;
  return plan;
}
int clusters_of(const UnitPlan& plan, int row_pairs) {
  return plan.n_whole + (row_pairs - plan.rp_tail0) * plan.groups * plan.nsplit;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// A pass with four pairs per cluster, run as persistent clusters of four pairs (one per resident slot)
// plus, on the SMs those leave idle (8-CTA clusters do not tile every GPC), persistent side clusters of
// two pairs and single-pair clusters sharing its work queue (WorkQueue).  The side launch follows the main
// one with programmatic stream serialisation: it starts once every main CTA is running, and completes
// after the main launch; the single-pair launch follows the side launch in the same way.  Taken when the
// pass has a queue word, the resident count is known and there are at least kCoRunMinWaves waves of main
// units; otherwise nothing is launched (*launched = false).
// The launches' reserves (see launch_corun) in quarters of the modelled ones, per pass.  Side clusters,
// measured at the long workload: x0.5 / x0.75 / x1 / x1.25 gave 37.8 / 37.8 / 39.9 / 39.9 ms for the
// grad_input pass and 40.5 / 40.6 / 40.0 / 40.3 ms for the grad_W pass (with single-pair side clusters);
// with two-pair side clusters x0.25 / x0.5 (grad_input) and x0.75 / x1 / x1.25 (grad_W) were all within
// 0.2 ms per step.  Single-pair clusters: x0.75 / x1 / x1.5 gave 36.94–36.98 / 36.93–36.98 / 37.64–37.81 ms
// for the grad_W pass; 0 launches none, as for the grad_input pass, whose single-pair units (two chunks
// over all the vocabulary blocks, ~12 ms each at the long workload) gained nothing: 36.95–37.27 ms with
// x1 and x1.5 against 36.76–36.79 without them.
constexpr int kReserveQuartersOnline = 2;
constexpr int kReserveQuartersGradW = 4;
constexpr int kReserveQuartersSingleOnline = 0;
constexpr int kReserveQuartersSingleGradW = 4;
// Side clusters that find no room beside the main clusters.  On the 152-SM GB300, 15 resident 8-CTA
// clusters leave 32 SMs idle; clusters that hold their SMs for a fixed time, launched one behind the other
// as here, showed room for 6 4-CTA clusters (two more start only once the 8-CTA clusters have finished)
// and then for 4 2-CTA clusters on the last 8 SMs (two groups of four, in neither of which a 4-CTA cluster
// is placed).  The single-pair launch starts only once every side CTA runs, so the side launch asks for
// the ones that fit.  On another layout a side cluster that finds no room delays the single-pair clusters
// to the end of the pass, where they find nothing left: the results are the same either way.
constexpr int kSideUnplaced = 2;

template <class MainKernel, class SideKernel, class SingleKernel>
cudaError_t launch_corun(MainKernel km, size_t smem_main, SideKernel ks, SingleKernel kx, size_t smem_side,
                         int res_main, const CUtensorMap& rows, const CUtensorMap& cols, const PairParams& p,
                         int h_chunks, int splits_option, int reserve_quarters, int reserve_quarters_single,
                         const DgPairArgs& a, cudaStream_t stream, bool* launched) {
  *launched = false;
  const int rp = row_pairs_of(p);
  const int P = p.P;
  const int S = side_pairs_for(P);
  const int main_groups = h_chunks / P;
  // (automatic scheduling only: splits_option 1 asks for one cluster per unit, k >= 2 for split units.  Four
  // pairs only: beside three-pair clusters (gemma2, 14 idle SMs, single-pair side clusters) the grad_W pass
  // gained 1.5% but the grad_input pass, with four waves of long units, lost 17% against its split tail;
  // beside two-pair clusters (8 idle SMs) nothing was gained.)
  if (a.work_q == nullptr || splits_option != 0 || P != 4 || res_main <= 0 || main_groups < 1 ||
      h_chunks % S != 0 || rp * main_groups < kCoRunMinWaves * res_main)
    return cudaSuccess;
  const int idle = device_sm_count() - 2 * P * res_main;
  int side = idle / (2 * S) - kSideUnplaced;
  if (side < 1) side = idle / (2 * S);
  if (side * S < 2) return cudaSuccess;
  const int single = (idle - 2 * S * side) / 2;   // single-pair clusters
  cudaError_t e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_main));
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_side))) !=
      cudaSuccess)
    return e;
  const UnitPlan plan = make_plan(rp, main_groups, (p.n_cols + kPN - 1) / kPN, 0, 1, 0, false);
  // A side unit (S pairs: the row pair's logits and S chunks' GEMM2) takes P (H + 256 S) / (S (H + 256 P))
  // times as long as a main unit (P pairs: the logits once and P chunks' GEMM2) at equal rates per pair, and
  // the same unit on a single pair (S times the logits and one chunk's GEMM2) S P (H + 256) / (H + 256 P)
  // times; each launch begins a row pair only while the main launch has that many units per main cluster
  // left, times its reserve quarters / 4 (measured per pass: the side pairs, with no hand-over to wait for,
  // run faster per pair than the model says in the grad_input pass).
  auto reserve_of = [&](long long quarters, long long time_num, long long time_den) {
    const long long num = quarters * time_num * res_main;
    const long long den = 4ll * time_den * main_groups;
    return static_cast<int>((num + den - 1) / den);
  };
  WorkQueue wq{a.work_q, a.side_count, a.single_count, a.single_units, kRoleMain, rp, main_groups, h_chunks / S, S,
               reserve_of(reserve_quarters, static_cast<long long>(P) * (p.H + S * kHc),
                          static_cast<long long>(S) * (p.H + P * kHc))};
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cm =
      cluster_config(dim3(2 * P * std::min(res_main, rp * main_groups), 1, 1), smem_main, P, stream, attr);
  if ((e = cudaLaunchKernelEx(&cm, km, rows, cols, p, a.status, plan, wq)) != cudaSuccess) return e;
  *launched = true;
  // the side and single-pair launches are an optimisation: without them the main clusters claim every unit
  // themselves (a launch that fails leaves the error cleared and the pass correct)
  PairParams ps = p;
  ps.P = S;
  WorkQueue wside = wq;
  wside.role = kRoleSide;
  cudaLaunchConfig_t cs = cluster_config(dim3(2 * S * side, 1, 1), smem_side, S, stream, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cs.numAttrs = 2;
  if (cudaLaunchKernelEx(&cs, ks, rows, cols, ps, a.status, plan, wside) != cudaSuccess) {
    (void)cudaGetLastError();
    return cudaSuccess;
  }
  if (single < 1 || reserve_quarters_single <= 0) return cudaSuccess;
  if (cudaFuncSetAttribute(kx, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_side)) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return cudaSuccess;
  }
  PairParams px = p;
  px.P = 1;
  WorkQueue wsingle = wq;
  wsingle.role = kRoleSingle;
  wsingle.reserve = std::max(wq.reserve, reserve_of(reserve_quarters_single, static_cast<long long>(S) * P * (p.H + kHc),
                                                    static_cast<long long>(p.H + P * kHc)));
  cudaLaunchAttribute attr1[2];
  cudaLaunchConfig_t cx = cluster_config(dim3(2 * single, 1, 1), smem_side, 1, stream, attr1);
  attr1[1] = attr[1];
  cx.numAttrs = 2;
  if (cudaLaunchKernelEx(&cx, kx, rows, cols, px, a.status, plan, wsingle) != cudaSuccess) (void)cudaGetLastError();
  return cudaSuccess;
}

}  // namespace

template <bool kVocabRows>
cudaError_t launch_dgrad_pair(const CUtensorMap& rows, const CUtensorMap& cols, const DgPairArgs& a,
                              cudaStream_t stream) {
  int h_chunks = 0;
  PairParams p = make_pair_params<kVocabRows>(a, &h_chunks);
  const bool filt = p.filter_eps > 0.f;
  static int res4 = 0;   // resident 8-CTA clusters of this pass's four-pair kernel
  if (res4 == 0 && !filt) {
    auto k4 = dgrad_pair_kernel<kVocabRows, false, kFourPairSlots>;
    const size_t s4 = pair_smem_bytes<kVocabRows, false, kFourPairSlots>();
    if (cudaFuncSetAttribute(k4, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s4)) == cudaSuccess)
      res4 = resident_clusters(k4, s4, 4, stream);
    else
      (void)cudaGetLastError();
  }
  if (four_pairs_with_side(p, h_chunks, kVocabRows ? a.token_splits : 0, a, res4)) p.P = 4;
  const bool four = p.P == 4;   // (exact passes only)
  const size_t smem = filt   ? pair_smem_bytes<kVocabRows, true>()
                      : four ? pair_smem_bytes<kVocabRows, false, kFourPairSlots>()
                             : pair_smem_bytes<kVocabRows, false>();
  auto kern = filt   ? dgrad_pair_kernel<kVocabRows, true, 2>
              : four ? dgrad_pair_kernel<kVocabRows, false, kFourPairSlots>
                     : dgrad_pair_kernel<kVocabRows, false, 2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int rp = row_pairs_of(p);
  const int nt = (p.n_cols + kPN - 1) / kPN;
  if (four && !filt) {
    bool launched = false;
    e = launch_corun(dgrad_pair_kernel<kVocabRows, false, kFourPairSlots, 1, true>, smem,
                     dgrad_pair_kernel<kVocabRows, false, 2, 2, true>, dgrad_pair_kernel<kVocabRows, false, 2, 4, true>,
                     pair_smem_bytes<kVocabRows, false>(), res4, rows, cols, p, h_chunks,
                     kVocabRows ? a.token_splits : 0, kVocabRows ? kReserveQuartersGradW : kReserveQuartersOnline,
                     kVocabRows ? kReserveQuartersSingleGradW : kReserveQuartersSingleOnline, a, stream, &launched);
    if (e != cudaSuccess || launched) return e;
  }
  UnitPlan plan = make_plan(rp, h_chunks / p.P, nt, 0, 1, 0, false);
  if (kVocabRows && a.split_scratch != nullptr) {
    // token-split tail of the grad_W pass: partial rows in the caller's scratch
    static int slots_of[2][kMaxPairs + 1] = {};
    int& slots = slots_of[filt ? 1 : 0][p.P];
    if (slots == 0) slots = resident_clusters(kern, smem, p.P, stream);
    const size_t per_su = sizeof(float) * 256 * (static_cast<size_t>(p.P) * kHc + 1);
    const int su_cap = static_cast<int>(std::min<size_t>(kMaxSplitUnits, a.split_scratch_bytes / per_su));
    plan = make_plan(rp, h_chunks / p.P, nt, slots, a.token_splits, su_cap, false);
    p.vs_o = a.split_scratch;
    p.vs_gb = a.split_scratch + static_cast<size_t>(su_cap) * 256 * p.P * kHc;
    p.vs_count = a.split_count;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(dim3(2 * p.P * clusters_of(plan, rp), 1, 1), smem, p.P, stream, attr);
  e = cudaLaunchKernelEx(&cfg, kern, rows, cols, p, a.status, plan, WorkQueue{});
  if (e != cudaSuccess) return e;
  if (kVocabRows && plan.nsplit > 1) {
    dw_vmerge_kernel<<<(rp - plan.rp_tail0) * 256, 128, 0, stream>>>(p, plan);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_dgrad_online(const CUtensorMap& hidden_map, const CUtensorMap& w_map, const DgPairArgs& a,
                                cudaStream_t stream) {
  int h_chunks = 0;
  PairParams p = make_pair_params<false>(a, &h_chunks);
  p.vs_mref = a.vs_mref;
  p.vs_part = a.vs_part;
  p.vs_stat = a.vs_stat;
  p.vs_o = a.vs_o;
  p.vs_count = a.vs_count;
  static int slots_of[kMaxPairs + 1] = {};
  if (slots_of[4] == 0) {
    auto k4 = dgrad_online_kernel<kFourPairSlots>;
    const size_t s4 = pair_smem_bytes<false, false, kFourPairSlots>();
    if (cudaFuncSetAttribute(k4, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s4)) == cudaSuccess)
      slots_of[4] = resident_clusters(k4, s4, 4, stream);
    else
      (void)cudaGetLastError();
  }
  if (four_pairs_with_side(p, h_chunks, a.vocab_splits, a, slots_of[4])) p.P = 4;
  const bool four = p.P == 4;
  const size_t smem = four ? pair_smem_bytes<false, false, kFourPairSlots>() : pair_smem_bytes<false, false>();
  auto kern = four ? dgrad_online_kernel<kFourPairSlots> : dgrad_online_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int rp = row_pairs_of(p);
  if (slots_of[p.P] == 0) slots_of[p.P] = resident_clusters(kern, smem, p.P, stream);
  if (four) {
    bool launched = false;
    e = launch_corun(dgrad_online_kernel<kFourPairSlots, 1, true>, smem, dgrad_online_kernel<2, 2, true>,
                     dgrad_online_kernel<2, 4, true>, pair_smem_bytes<false, false>(), slots_of[4], hidden_map, w_map,
                     p, h_chunks, a.vocab_splits, kReserveQuartersOnline, kReserveQuartersSingleOnline, a, stream,
                     &launched);
    if (e != cudaSuccess || launched) return e;
  }
  // vocabulary-split tail: the accumulators go to the split scratch (16 MiB),
  // or to grad_W when it is larger and holds nothing yet (written only by the grad_W pass, after the merge)
  const size_t per_su = sizeof(float) * 256 * p.P * kHc;
  size_t scratch = a.vs_o == nullptr ? 0 : kSplitAccBytes;
  if (a.vs_o != nullptr && a.grad_W != nullptr && !a.accumulate &&
      sizeof(float) * static_cast<size_t>(a.V) * a.H > scratch) {
    scratch = sizeof(float) * static_cast<size_t>(a.V) * a.H;
    p.vs_o = a.grad_W;
  }
  const int su_cap = static_cast<int>(std::min<size_t>(kMaxSplitUnits, scratch / per_su));
  const UnitPlan plan =
      make_plan(rp, h_chunks / p.P, (p.n_cols + kPN - 1) / kPN, slots_of[p.P], a.vocab_splits, su_cap, true);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(dim3(2 * p.P * clusters_of(plan, rp), 1, 1), smem, p.P, stream, attr);
  e = cudaLaunchKernelEx(&cfg, kern, hidden_map, w_map, p, a.status, plan, WorkQueue{});
  if (e != cudaSuccess) return e;
  if (plan.nsplit > 1) {
    online_vmerge_kernel<<<(rp - plan.rp_tail0) * 256, 128, 0, stream>>>(p, plan);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_dgrad_both(const CUtensorMap& hidden_map, const CUtensorMap& w_map, const DgPairArgs& a,
                              cudaStream_t stream) {
  int hc_in = 0, hc_w = 0;
  const PairParams p_in = make_pair_params<false>(a, &hc_in);
  const PairParams p_w = make_pair_params<true>(a, &hc_w);
  if (p_in.P != p_w.P) {
    // different cluster shapes: two launches (the queue word, if any, is the grad_W pass's)
    DgPairArgs ai = a;
    ai.work_q = nullptr;
    cudaError_t e = launch_dgrad_pair<false>(hidden_map, w_map, ai, stream);
    if (e != cudaSuccess) return e;
    return launch_dgrad_pair<true>(w_map, hidden_map, a, stream);
  }
  const bool filt = a.filter_eps > 0.f;
  const bool four = p_in.P == 4;
  const size_t smem = filt   ? std::max(pair_smem_bytes<false, true>(), pair_smem_bytes<true, true>())
                      : four ? std::max(pair_smem_bytes<false, false, kFourPairSlots>(), pair_smem_bytes<true, false, kFourPairSlots>())
                             : std::max(pair_smem_bytes<false, false>(), pair_smem_bytes<true, false>());
  auto kern = filt ? dgrad_both_kernel<true, 2> : four ? dgrad_both_kernel<false, kFourPairSlots> : dgrad_both_kernel<false, 2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int in_rp = row_pairs_of(p_in), w_rp = row_pairs_of(p_w);
  const int n_in = in_rp * (hc_in / p_in.P);
  const int n_w = w_rp * (hc_w / p_w.P);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(dim3(2 * p_in.P * (n_in + n_w), 1, 1), smem, p_in.P, stream, attr);
  e = cudaLaunchKernelEx(&cfg, kern, hidden_map, w_map, p_in, p_w, a.status, n_in, in_rp, w_rp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template cudaError_t launch_dgrad_pair<false>(const CUtensorMap&, const CUtensorMap&, const DgPairArgs&, cudaStream_t);
template cudaError_t launch_dgrad_pair<true>(const CUtensorMap&, const CUtensorMap&, const DgPairArgs&, cudaStream_t);

}  // namespace flce
