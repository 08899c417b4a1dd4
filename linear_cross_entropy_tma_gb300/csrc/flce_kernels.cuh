// flce_kernels.cuh -- workspace layout and launchers of the fused linear cross-entropy kernels.
//
// Pass structure of one flce_fwd_bwd call in the classic flow (all on one stream, no host
// synchronisation; the default flow replaces steps 1-4 by the online grad_input pass, see flce_launch.cu):
//   1. lse_partial   logits tile GEMM (tcgen05, TMEM accumulators, TMA-fed) per (128-token tile,
//                    vocabulary split); the epilogue keeps an online per-row (max, sum-exp) over the
//                    split's 256-wide vocabulary tiles and picks up the target logit z_y.
//   2. lse_merge     per row: log-sum-exp merge of the split partials -> LSE, per-row loss term,
//                    per-row statistics used by the backward passes.
//   3. loss_reduce   one CTA: deterministic sum of the per-row terms, the valid count and the scale
//                    s = 1/max(n_valid, 1) (mean) or 1 (sum).
//   4. dgrad<tokens> grad_input: per (128-token tile, H chunk) recompute logits tiles over all of V,
//                    form dlogits in registers, stage it as bf16 in shared memory and feed it to a
//                    second tcgen05 GEMM that accumulates grad_input in TMEM.
//   5. dgrad<vocab>  grad_W (+ grad_bias): per (128-row vocabulary tile, H chunk) the same over all
//                    tokens, accumulating grad_W in TMEM in fp32.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace flce {

constexpr int kMaxSplits = 32;     // vocabulary splits of the LSE pass
constexpr int kTileM = 128;        // rows of every MMA tile (tokens or vocabulary rows)

// Accumulator scratch of the vocabulary-split units of the online grad_input pass (16 MiB).
constexpr size_t kSplitAccBytes = size_t(16) << 20;
// Vocabulary-split work units of the online grad_input pass (see launch_dgrad_online): at most this many,
// their accumulators in the split scratch (or in grad_W, see launch_dgrad_online), their row sums in vs_*.
constexpr int kMaxSplitUnits = 64;

struct FusedWorkspace {
  uint32_t* status;  // header: status word
  float* scale;      // header: gradient scale G = grad_scale / max(n_valid, 1) (mean) or grad_scale
  int64_t* n_valid;  // header: valid count
  uint32_t* skipped; // header: dS halves whose GEMM2 the gradient filter skipped (both passes)
  uint32_t* fallback; // header: non-zero when the online grad_input pass handed the call to the classic passes
  uint32_t* vs_count; // header: vocabulary-split clusters of the online grad_input pass
  uint32_t* ts_count; // header: token-split clusters of the grad_W pass
  unsigned long long* work_q;  // header: [2] work queues of the grad_input and grad_W passes (zeroed per call)
  uint32_t* side_count;        // header: [2] launches of side clusters beside the four-pair clusters, and
                               // side clusters that took at least one unit
  uint32_t* single_units;      // header: [2] units the single-pair clusters took in the grad_input and
                               // grad_W passes
  uint32_t* single_count;      // header: [2] launches of single-pair clusters, and single-pair clusters
                               // that took at least one unit
  uint32_t* zf_neg;  // header: non-zero when the log form of dS does not apply (some valid row has
                     // f u <= 0 with u its upstream gradient, or the gradient scale is <= 0)
  float2* part;      // [kMaxSplits][BTp] (max in log2 units, sum of 2^(x - max)); free again by the
                     // grad_W pass, which keeps the partial rows of its token-split units there
  size_t part_bytes;
  float* part_t;     // [kMaxSplits][BTp] sum of 2^(x - max) z (only when the entropy is requested)
  float* zy;         // [BTp] target logit
  float4* stats;     // [BT rounded up to 256] per row t, with LSE2 = LSE log2 e, f = 1 + 2 z_loss LSE and u
                     // the row's upstream gradient (1 unless reduction none):
                     //   x = log2(f u) - LSE2 (-inf for ignored rows and when f u <= 0), y = target as int bits
                     //   (-1 for ignored rows), z = valid ? u : 0, w = LSE2; rows past BT: (-inf, -1, 0, 0)
  float2* stats_ct;  // [BT rounded up to 256] the first two words of stats (x, y): what the exact grad_W pass
                     // stages per block
  float* row_loss;   // [BTp] valid * (LSE - z_y + z_loss LSE^2)
  float* colb2;      // [V rounded up to 256] bias * log2 e (0 without bias); -inf past V
  uint32_t* row_redo; // [BTp] online flow: 1 for a row the grad_input pass left to the classic passes
  float* vs_mref;    // [kMaxSplitUnits][256] online pass, vocabulary-split units: per-row reference
  float4* vs_part;   // [kMaxSplitUnits][256][4][2] their pairs' partial sums
  float4* vs_stat;   // [kMaxSplitUnits][256] their row sums
  float* split_acc;  // [kSplitAccBytes] accumulators of the online pass's vocabulary-split units
};

size_t fused_workspace_bytes(int64_t BT, int64_t V);
FusedWorkspace carve_workspace(void* base, int64_t BT, int64_t V);

// Scratch of the vocabulary sort (vocab_sort.cu), placed after the fused workspace when requested.
struct VocabSortWorkspace {
  float* col_part;      // [64][H] partial column sums of hidden
  float* hbar;          // [H] mean of the hidden rows
  float* logit_avg;     // [V] average logit per vocabulary entry
  uint32_t* keys[2];    // [V] radix keys (double buffer)
  int32_t* vals[2];     // [V] vocabulary indices (double buffer); vals[0] ends as the sorted order
  uint32_t* hist;       // [ceil(V / 8192)][256] per-block digit counts / offsets
  int32_t* inv;         // [V] sorted position of each vocabulary entry
  float* bias;          // [V] bias in sorted order
  int64_t* target;      // [BT] targets as sorted positions (-1: ignored or out of range)
  uint16_t* W;          // [V][H] W in sorted row order
};
size_t vocab_sort_workspace_bytes(int64_t BT, int64_t H, int64_t V);
VocabSortWorkspace carve_vocab_sort(void* base, int64_t BT, int64_t H, int64_t V);

struct FusedArgs {
  const uint16_t* hidden;
  const uint16_t* W;
  const float* bias;
  const int64_t* target;
  int64_t BT, H, V;
  int64_t ignore_index;
  int reduction;              // 0 mean, 1 sum, 2 none
  float z_loss;
  float* loss;                // may be NULL for reduction none
  uint16_t* grad_input;
  float* grad_W;
  float* grad_bias;
  int64_t* n_valid_out;
  float grad_scale;           // upstream gradient of the reduced loss
  const float* grad_tok;      // reduction none: upstream gradient per token, or NULL (ones)
  float* loss_tok;            // per-token losses out, or NULL
  float* entropy;             // per-row entropy of softmax(z) out, or NULL
  float filter_eps;           // > 0: gradient filtering threshold
  bool accumulate;            // gradients += instead of =
  bool sort_vocab;            // run the passes on the vocabulary sorted by average logit
  float* logit_avg_out;       // [V] average logit per vocabulary entry out, or NULL (needs sort_vocab)
  int32_t* vocab_order_out;   // [V] sorted order out, or NULL (needs sort_vocab)
  bool separate_lse;          // always the classic flow (LSE tiles first)
  int vocab_splits;           // online grad_input pass: 0 automatic, 1 never, k >= 2 every row block in k parts
  int token_splits;           // grad_W pass: the same over token ranges
  uint32_t debug_stall_us;    // test-only: the gradient passes' producers first wait this long on nothing
};

// The vocabulary sort: logit_avg, the sorted order (in w.vals[0]), the sorted copies of W, the bias and
// the targets.  Bad targets set the status bit here.
cudaError_t launch_vocab_sort(const FusedArgs& a, const VocabSortWorkspace& w, uint32_t* status, int num_sms,
                              cudaStream_t stream);

// Arguments of the gradient passes on CTA pairs (flce_bwd.cu).
struct DgPairArgs {
  const float* bias;
  const float4* stats;
  const float2* stats_ct;    // (x, y) of stats, compact
  const float* colb2;
  const float* scale;
  const uint32_t* zf_neg;
  float z_loss;
  bool accumulate;
  float filter_eps;
  uint32_t* skip_count;
  const int32_t* row_perm;   // grad_W pass: output row of each (sorted) vocabulary row, or NULL
  int BT, V, H;
  uint16_t* grad_input;
  float* grad_W;
  float* grad_bias;
  uint32_t* status;
  const uint32_t* gate;      // non-NULL: the launch does nothing unless *gate != 0
  // grad_input pass without a prior LSE pass (launch_dgrad_online)
  const int64_t* target;
  int64_t ignore_index;
  const float* grad_tok;
  const uint16_t* Wmat;
  float* mref_g;             // [BT rounded up to 256]
  float4* part_g;            // [BT rounded up to 256][4][2]
  float* entropy_out;        // per-row entropy out, or NULL
  uint32_t* row_redo;        // [BTp] rows the online pass left to the classic one (see flce_bwd.cu)
  float4* stats_out;
  float2* stats_ct_out;
  float* row_loss;
  float* loss_tok;
  uint32_t* zf_neg_out;
  uint32_t* fallback;
  // vocabulary-split units of the online pass: 0 = split the last, partly filled wave automatically,
  // 1 = never, k >= 2 = every row block into (up to) k parts; their scratch (null: no splitting)
  int vocab_splits;
  float* vs_mref;
  float4* vs_part;
  float4* vs_stat;
  float* vs_o;
  uint32_t* vs_count;
  // token-split units of the grad_W pass (same meaning as vocab_splits); their partial rows go to
  // split_scratch (null: no splitting)
  int token_splits;
  float* split_scratch;
  size_t split_scratch_bytes;
  uint32_t* split_count;
  uint32_t debug_stall_us;   // test-only (flce_fwd_bwd_options.debug_stall_us)
  // Shared work queue (a zeroed 64-bit word) for a pass run by persistent clusters of four pairs plus
  // launches of smaller side and single-pair clusters on the SMs they leave idle, or NULL (one cluster
  // per unit); side_count / single_count: [2] incremented once per side (single-pair) launch, and once
  // per side (single-pair) cluster that took a unit; single_units: this pass's units taken by single-pair
  // clusters (workspace header)
  unsigned long long* work_q;
  uint32_t* side_count;
  uint32_t* single_count;
  uint32_t* single_units;
};

// kVocabRows = false: grad_input pass (rows = tokens, reduction over the vocabulary);
// true: grad_W / grad_bias pass (rows = vocabulary entries, reduction over tokens).
// rows / cols: tensor maps with 128-row x 64-column boxes of the row and column matrices.
template <bool kVocabRows>
cudaError_t launch_dgrad_pair(const CUtensorMap& rows, const CUtensorMap& cols, const DgPairArgs& a,
                              cudaStream_t stream);

// The grad_input pass without a prior LSE pass: online softmax over the vocabulary against a fixed per-row
// reference (the row's largest logit in the first 128 columns), which also produces the per-token
// statistics, the loss terms and zf_neg for the grad_W pass and the loss reduction.  Needs the gradient
// scale (ws.scale) and the bias table (colb2) in place.  Sets *fallback when some row's sum leaves the safe
// range; the classic passes, gated on it, then redo the call.
cudaError_t launch_dgrad_online(const CUtensorMap& hidden_map, const CUtensorMap& w_map, const DgPairArgs& a,
                                cudaStream_t stream);

// Both gradient passes, as one launch when they have the same cluster shape (the grad_W pass's clusters
// then fill the SMs the grad_input pass's last wave leaves idle), else as two.  hidden_map / w_map: the
// 128-row x 64-column box maps of hidden and W.
cudaError_t launch_dgrad_both(const CUtensorMap& hidden_map, const CUtensorMap& w_map, const DgPairArgs& a,
                              cudaStream_t stream);

// Encodes a 2-D bf16 tensor map (rows x cols, row-major) with a box of box_rows x 64 columns and
// 128-byte swizzle.  Returns false (and fills err) when the driver refuses the descriptor.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    char* err, size_t err_len);

// Enqueues every pass.  Returns cudaSuccess or the first launch error; tensor-map failures are
// reported as cudaErrorInvalidValue with a message in err.
// events: NULL, or 5 caller-owned events recorded at the pass boundaries (see flce_fwd_bwd_timed).
cudaError_t launch_fused(const FusedArgs& a, void* workspace, int num_sms, cudaStream_t stream, char* err,
                         size_t err_len, cudaEvent_t const* events = nullptr);

}  // namespace flce
