/*
 * flce.h -- C ABI of the GB300 (sm_103a) fused linear cross-entropy library, libflce.so.
 *
 * Two operations:
 *
 *   flce_fwd_bwd   Fused LM-head cross-entropy.  With logits z = hidden . W^T (+ bias) it returns
 *                  the loss and the gradients grad_input = dlogits . W, grad_W = dlogits^T . hidden
 *                  and grad_bias = sum_t dlogits[t, :], where
 *                      dlogits[t, :] = s * [y_t valid] * (softmax(z_t) * (1 + 2 z_loss LSE_t) - onehot(y_t))
 *                  and s = 1 / max(n_valid, 1) for the mean reduction, 1 for the sum reduction.
 *                  The (BT, V) logits are never written to device memory: each logits tile lives
 *                  only in tensor memory and registers of the CTA that computes it.
 *                  Definitions: "Fused Linear Cross-Entropy: The Math, the Memory Wall, and Two Ways
 *                  Around It", sections "The setting" (loss), "The identity that makes fused fwbw
 *                  possible" (softmax - onehot, two-scalar LSE) and "From dlogits to grad_input and
 *                  grad_W" (the two boxed GEMMs and the bias column sum).  The z-loss term
 *                  z_loss * LSE^2 per valid token follows "Greyhound -- Cross-Entropy", formulas and
 *                  "Loss and gradient together".
 *
 *   ce_with_grad   Row-wise cross-entropy over logits that already exist, in place: the logits buffer
 *                  is overwritten with dlogits = [y valid] * (softmax * (1 + 2 z_loss LSE) - onehot),
 *                  and the sums ce_sum = sum_valid (LSE - z_y), z_sum = sum_valid LSE^2 and the count
 *                  n_valid are returned ("Greyhound -- Cross-Entropy", "Kernel design", "Shape and
 *                  dtype constraints" and the raw helper under "Usage").
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device, row-major and contiguous.
 *     bf16 tensors are passed as uint16_t (raw bfloat16 bit patterns).
 *   - The caller owns and allocates every buffer, including the workspace.  The library keeps no
 *     state between calls (beyond a per-process cache of how many clusters of each shape the device
 *     holds at once) and touches no memory other than the buffers it is given.  (flce_fwd_bwd may use
 *     grad_W as scratch before writing it, when the call does not accumulate.)
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and the call
 *     returns without synchronising.  Only flce_read_device_status synchronises the stream.  A call
 *     can be captured into a CUDA graph and replayed; the occupancy query behind the cache is not made
 *     while the stream is capturing (that call then plans no split tails, see vocab_splits).
 *   - Outputs are overwritten (flce_fwd_bwd_ex can accumulate into them instead).
 *   - Argument errors are reported synchronously by the return code before anything is enqueued.
 *     Data errors (a target outside [0, V) that is not ignore_index) are found on the device: the
 *     row is treated as ignored and bit FLCE_STATUS_BAD_TARGET is set in the workspace status word.
 *   - Every wait inside a kernel is bounded; a wait that gives up sets FLCE_STATUS_TIMEOUT in the
 *     status word and the kernel returns instead of hanging.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum flce_status {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,          /* null required pointer, negative size, bad reduction, bias /
                                        grad_bias mismatch, aliasing outputs */
  FLCE_ERR_MISALIGNED = 2,           /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the matching *_workspace_size() */
  FLCE_ERR_UNSUPPORTED = 4,          /* a size outside what the kernels handle (see each call) */
  FLCE_ERR_CUDA = 5,                 /* a CUDA runtime call or a kernel launch failed */
  FLCE_ERR_NO_DEVICE = 6             /* the current device is not a compute capability 10.3 GPU */
} flce_status;

/* reduction argument of flce_fwd_bwd */
#define FLCE_REDUCTION_MEAN 0
#define FLCE_REDUCTION_SUM 1
#define FLCE_REDUCTION_NONE 2  /* per-token losses; flce_fwd_bwd_ex only */

/* bits of the device status word (first 4 bytes of either workspace) */
#define FLCE_STATUS_BAD_TARGET 0x1u
#define FLCE_STATUS_TIMEOUT 0x2u
#define FLCE_STATUS_INTERNAL 0x4u   /* a self-check of the vocabulary sort failed (a defect; results invalid) */

/*
 * Bytes of workspace flce_fwd_bwd needs for these sizes (O(BT + V) floats: per-row LSE statistics,
 * per-row loss terms, the per-column bias in log2 units, the status word and the valid count; plus a
 * fixed 16 MiB for the accumulators of the grad_input pass's vocabulary-split clusters).
 * Returns 0 for negative sizes.
 */
size_t flce_workspace_size(int64_t BT, int64_t H, int64_t V);

/*
 * Fused linear cross-entropy, forward and backward in one call.
 *
 *   hidden      [BT, H] bf16, device.                      (p1 "The setting": hidden[t] in R^H)
 *   W           [V, H]  bf16, device.                      (LM-head weight, V x H)
 *   bias        [V] fp32, device, or NULL for no bias.
 *   target      [BT] int64, device: class index in [0, V), or ignore_index.
 *   BT, H, V    sizes.  BT >= 0; H >= 8 with H % 8 == 0 (16-byte rows for the tensor-memory-access
 *               copies); V >= 1.  BT, V < 2^31.  Otherwise FLCE_ERR_UNSUPPORTED / INVALID_ARG.
 *   ignore_index  rows whose target equals it contribute nothing (PyTorch's -100 by default).
 *   reduction   FLCE_REDUCTION_MEAN (divide by max(n_valid, 1)) or FLCE_REDUCTION_SUM.
 *   z_loss      multiplier of the per-token LSE^2 term (0 disables it).
 *   loss        [1] fp32, device: the reduced loss.
 *   grad_input  [BT, H] bf16, device, or NULL to skip the grad_input pass.
 *   grad_W      [V, H] fp32, device, or NULL.
 *   grad_bias   [V] fp32, device, or NULL; must be NULL when bias is NULL.
 *               When both grad_W and grad_bias are NULL the grad_W pass is skipped.
 *   n_valid     [1] int64, device, or NULL: number of rows whose target is in [0, V).
 *   workspace   device scratch of at least flce_workspace_size(BT, H, V) bytes, 256-byte aligned.
 *               Its contents on entry do not matter.  Overlapping calls must use separate
 *               workspaces.
 *   stream      cudaStream_t.
 *
 * hidden, W, grad_input: 16-byte aligned.  bias, target, grad_W, grad_bias, loss: 4/8-byte aligned
 * (natural alignment).
 */
flce_status flce_fwd_bwd(const uint16_t* hidden, const uint16_t* W, const float* bias,
                         const int64_t* target, int64_t BT, int64_t H, int64_t V,
                         int64_t ignore_index, int reduction, float z_loss, float* loss,
                         uint16_t* grad_input, float* grad_W, float* grad_bias, int64_t* n_valid,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * flce_fwd_bwd with timing hooks: identical work and results, plus cudaEventRecord of caller-created
 * CUDA events at the pass boundaries on `stream`, so a caller can time each kernel inside a longer
 * timed region without any synchronisation:
 *   events[0] before the LSE pass        events[1] after the LSE tile kernel
 *   events[2] after the merge + loss reduction
 *   events[3] after the grad_input pass  events[4] after the grad_W pass
 * in the classic flow; when the grad_input pass finds the LSE itself (the default whenever grad_input is
 * requested, see flce_fwd_bwd_options.separate_lse_pass, which this call does not take):
 *   events[1] after the bias table and the valid count   events[2] after that grad_input pass
 *   events[3] after the loss reduction and the gated classic kernels   events[4] after the grad_W pass
 * (a skipped pass records its two events back to back; when both gradient passes run as one launch,
 * which they do whenever both are requested and have the same cluster shape, events[3] is recorded
 * together with events[4], after that launch).  n_events must be 0 or 5; events may be
 * NULL when n_events is 0.  The events are owned by the caller (cudaEvent_t handles).
 */
flce_status flce_fwd_bwd_timed(const uint16_t* hidden, const uint16_t* W, const float* bias,
                               const int64_t* target, int64_t BT, int64_t H, int64_t V,
                               int64_t ignore_index, int reduction, float z_loss, float* loss,
                               uint16_t* grad_input, float* grad_W, float* grad_bias,
                               int64_t* n_valid, void* workspace, size_t workspace_bytes,
                               void* stream, void* const* events, int n_events);

/*
 * Options of flce_fwd_bwd_ex (all zero / NULL except grad_scale = 1 reproduces flce_fwd_bwd).
 *
 * The loss gradient is scaled by the upstream gradient as in "Cut Cross Entropy visualized",
 * "Breakdown: Backward Pass", step 4 (the d_out * grad_scale factor); for an unreduced loss the upstream
 * gradient has one entry per token (PyTorch's convention for reduction='none').
 *
 *   grad_scale           multiplies every gradient (the upstream gradient of the reduced loss).
 *                        Any finite value; 0 gives zero gradients.  Does not change the loss.
 *   grad_loss_per_token  [BT] fp32, device, or NULL (all ones): with FLCE_REDUCTION_NONE, the upstream
 *                        gradient g_t of token t's loss; the gradients are those of
 *                        grad_scale * sum_t g_t l_t.  Must be NULL for MEAN and SUM.
 *   loss_per_token       [BT] fp32, device, or NULL: receives l_t = LSE_t - z_y + z_loss LSE_t^2 on
 *                        valid rows and 0 on ignored rows (any reduction).
 *   accumulate           non-zero: grad_input, grad_W and grad_bias receive += instead of = (their
 *                        previous contents are added to; grad_input is re-rounded to bf16).
 *   entropy              [BT] fp32, device, or NULL: the entropy of softmax(z_t) for every row,
 *                        -sum_n p_n log p_n = LSE_t - sum_n p_n z_n (verl's per-row entropy output,
 *                        "Fused Linear Cross-Entropy", "Strategy 2"), ignored rows included.  Costs
 *                        one more multiply-add per logit in the LSE pass.
 *   filter_eps           0 (exact) or a positive threshold: the gradient-filtering variant of "Cut Cross
 *                        Entropy visualized", "Gradient filtering", applied as there to the unscaled
 *                        gradient p f - onehot (before the upstream gradient and the mean scale).  A
 *                        256-row x 128-column block of dS (two CTAs' 128 rows; tokens x vocabulary in
 *                        the grad_input pass, vocabulary x tokens in the grad_W pass) whose unscaled
 *                        entries are all at most filter_eps in magnitude adds nothing to grad_input /
 *                        grad_W (its tensor-core GEMM is skipped).  grad_bias and the loss stay exact.
 *                        Error bound: each element of grad_input (grad_W) differs from the exact
 *                        gradient by at most the sum of |dS| |W| (|dS| |hidden|) over the entries whose
 *                        unscaled magnitude is at most filter_eps, plus the usual rounding.
 *                        The number of skipped blocks is the 32-bit word at byte 20 of the workspace.
 *   sort_vocab           non-zero: the vocabulary sort of "Cut Cross Entropy visualized", "Vocabulary
 *                        Sorting", which makes filtering skip more blocks.  logit_avg[n], the mean of
 *                        z[t, n] over all BT rows (ignored rows included; "Forward pass"), is computed
 *                        as W[n] . mean_t hidden[t] + b[n]; every pass then runs on the vocabulary in
 *                        decreasing logit_avg order (equal keys by index).  Results are those of the
 *                        unsorted call up to rounding order; the filter's error bound is unchanged.
 *                        Needs flce_workspace_size_ex(BT, H, V, options) bytes of workspace (adds a
 *                        sorted copy of W: V x H bf16).
 *   logit_avg            [V] fp32, device, or NULL: receives logit_avg (requires sort_vocab).
 *   vocab_order          [V] int32, device, or NULL: receives the sorted order, entry k = the vocabulary
 *                        index at sorted position k (requires sort_vocab).
 *   separate_lse_pass    non-zero: compute every row's LSE in a pass of its own before the gradient passes
 *                        (the two-pass scheme of "Cut Cross Entropy visualized", "Backward pass").  By
 *                        default, when grad_input is requested, the grad_input pass finds the LSE itself
 *                        (and the entropy, when requested) (online softmax against a per-row
 *                        reference, "Fused Linear Cross-Entropy", "Strategy 2"), one GEMM over the logits
 *                        fewer; rows whose sums leave that pass's safe range are redone with the separate
 *                        pass, on the device.  Both give the same results up to rounding.
 *                        With filter_eps > 0 that grad_input pass is exact and only the grad_W pass
 *                        filters (a result within the same bound).
 *   vocab_splits         work split of that grad_input pass (default flow only).  0: automatic -- the
 *                        row blocks of its last, partly filled wave of clusters (all of them when
 *                        they fill less than a wave: small BT) are each split into vocabulary ranges
 *                        processed by separate clusters, whose partial sums (against their own
 *                        references) a merge kernel rescales and adds ("Cut Cross Entropy visualized",
 *                        "Triton kernel, online softmax across vocab splits"); 1: never split; k >= 2:
 *                        split every row block into up to k ranges (fewer when the scratch, 64 split
 *                        clusters, or ranges of at least 4 x 256 columns do not allow k; at most 16).
 *                        Results are the same up to rounding order.  Negative:
 *                        FLCE_ERR_INVALID_ARG.  The number of vocabulary-split clusters the call ran is
 *                        the 32-bit word at byte 28 of the workspace.
 *                        With 0, a pass that runs four pairs per cluster (clusters of 8 CTAs) over at
 *                        least three waves of work units is scheduled instead as persistent 8-CTA
 *                        clusters that take units from a queue in the workspace header, plus a second
 *                        launch of 4-CTA clusters (two pairs), started by programmatic dependent launch,
 *                        on the SMs the 8-CTA clusters leave idle, and (grad_W pass) behind it a third
 *                        launch of 2-CTA clusters (one pair) on the SMs where no 4-CTA cluster is placed.  Both take two
 *                        256-column H chunks of the last row blocks at a time (the 4-CTA clusters
 *                        computing those blocks' logits once per two chunks, the 2-CTA clusters once per
 *                        chunk, one chunk after the other) and stop early enough to finish with the
 *                        8-CTA clusters.  No unit is split then, and the results are bit for bit those of
 *                        one 8-CTA cluster per unit.  Each pass that did this adds 1 to the word at byte
 *                        56 of the workspace, and 1 to the word at byte 72 when it also launched 2-CTA
 *                        clusters; the words at bytes 60 and 76 count the 4-CTA and 2-CTA clusters that
 *                        took work, and those at bytes 64 and 68 the units the 2-CTA clusters took in the
 *                        grad_input and the grad_W pass.
 *   token_splits         the same for the grad_W pass, whose clusters own vocabulary rows and run over
 *                        the tokens: 0 splits the row blocks of its last, partly filled wave into token
 *                        ranges (partial grad_W / grad_bias rows, added in order by a merge kernel), 1
 *                        never, k >= 2 every row block into up to k ranges (within the workspace's
 *                        scratch: fewer at small BT).  The classic flow's single launch of both passes
 *                        (separate_lse_pass with grad_input and grad_W) does not split.  The number of
 *                        token-split clusters is the word at byte 32 of the workspace.  0 also allows
 *                        the persistent scheduling with 4-CTA clusters beside the 8-CTA ones described
 *                        under vocab_splits.
 *   debug_stall_us       test-only; 0 in normal use.  When > 0 (at most 1000000, else
 *                        FLCE_ERR_INVALID_ARG), the TMA producer of every CTA of the gradient passes first
 *                        waits this many microseconds for an mbarrier phase that nothing completes, before
 *                        it issues any copy.  That wait gives up as any bounded wait in the kernels does:
 *                        it raises the CTA's abort flag, every role of the cluster winds down (nothing is
 *                        in flight), TMEM is freed, the kernel sets FLCE_STATUS_TIMEOUT in the status word
 *                        and returns.  The rest of the call still runs; its results are invalid.  This is
 *                        how the timeout path (the bounded replacement of the spin lock in "Cut Cross
 *                        Entropy visualized", "Forward kernel") is exercised without faulting or hanging
 *                        a GPU; the next call on the same stream and workspace is unaffected.
 */
typedef struct flce_fwd_bwd_options {
  float grad_scale;
  const float* grad_loss_per_token;
  float* loss_per_token;
  int accumulate;
  float* entropy;
  float filter_eps;
  int sort_vocab;
  float* logit_avg;
  int32_t* vocab_order;
  int separate_lse_pass;
  int vocab_splits;
  int token_splits;
  uint32_t debug_stall_us;
} flce_fwd_bwd_options;

/* Bytes of workspace flce_fwd_bwd_ex needs with these options (NULL: flce_workspace_size). */
size_t flce_workspace_size_ex(int64_t BT, int64_t H, int64_t V, const flce_fwd_bwd_options* options);

/*
 * flce_fwd_bwd with options (NULL options = the defaults above).  reduction may also be
 * FLCE_REDUCTION_NONE; then `loss` may be NULL and, when given, receives the plain sum of the
 * per-token losses.  Pointer alignment: loss_per_token, grad_loss_per_token, entropy, logit_avg and
 * vocab_order 4 bytes.
 */
flce_status flce_fwd_bwd_ex(const uint16_t* hidden, const uint16_t* W, const float* bias,
                            const int64_t* target, int64_t BT, int64_t H, int64_t V,
                            int64_t ignore_index, int reduction, float z_loss, float* loss,
                            uint16_t* grad_input, float* grad_W, float* grad_bias, int64_t* n_valid,
                            void* workspace, size_t workspace_bytes,
                            const flce_fwd_bwd_options* options, void* stream);

/* Bytes of workspace ce_with_grad needs for B rows (per-row partial sums and the status word). */
size_t ce_workspace_size(int64_t B, int64_t V);

/*
 * Standalone cross-entropy with the logits gradient written in place.
 *
 *   logits      [B, V] bf16, device, 16-byte aligned.  In: logits.  Out: dlogits (bf16).
 *   labels      [B] int64, device.
 *   B, V        B >= 0, 1 <= V < 2^31.
 *   ignore_index  rows with this label: no loss, not counted, gradient row written as zeros.
 *   z_loss      multiplier used in the gradient; z_sum itself is returned unscaled.
 *   ce_sum      [1] fp32, device: sum over valid rows of LSE - z_y.
 *   z_sum       [1] fp32, device: sum over valid rows of LSE^2.
 *   n_valid     [1] int64, device: number of valid rows.
 *               The mean loss of p3 "Usage" is ce_sum / max(n_valid, 1).
 *   workspace   at least ce_workspace_size(B, V) bytes, 256-byte aligned.
 */
flce_status ce_with_grad(uint16_t* logits, const int64_t* labels, int64_t B, int64_t V,
                         int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum,
                         int64_t* n_valid, void* workspace, size_t workspace_bytes, void* stream);

/* element types of the standalone CE's logits */
#define FLCE_DTYPE_BF16 0
#define FLCE_DTYPE_F16 1
#define FLCE_DTYPE_F32 2

/*
 * ce_with_grad for bf16, fp16 or fp32 logits ("Greyhound -- Cross-Entropy", "Shape and dtype
 * constraints"), with the gradient in place, into a separate buffer (the non-mutating form of the
 * functional wrapper in "Usage"), or not at all.
 *
 *   logits      [B, V] of `dtype`, device, 16-byte aligned.  Read only, unless dlogits == logits.
 *   dlogits     [B, V] of `dtype`, device, 16-byte aligned: == logits (in place, exactly ce_with_grad for
 *               bf16), a separate buffer that must not overlap the logits (the logits are left
 *               unchanged), or NULL (ce_sum, z_sum and n_valid only; no gradient is written).
 *   dtype       FLCE_DTYPE_BF16, FLCE_DTYPE_F16 or FLCE_DTYPE_F32.
 * The other arguments, the results and the errors are those of ce_with_grad; the arithmetic is fp32
 * for every dtype and dlogits is rounded to nearest-even in the logits' type.
 */
flce_status ce_with_grad_ex(const void* logits, void* dlogits, int dtype, const int64_t* labels, int64_t B,
                            int64_t V, int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum,
                            int64_t* n_valid, void* workspace, size_t workspace_bytes, void* stream);

/*
 * ce_with_grad without a workspace, for callers that cannot allocate device memory.
 * (No counterpart on the pages: an addition of this library.)
 *
 * Some callers are never allowed to call cudaMalloc themselves: a plugin inside an engine whose
 * device memory is planned ahead and which receives only its input and output buffers, or a
 * service that forbids allocation after start-up because an allocation can block or fail at run
 * time.  This call does the same work as ce_with_grad (same kernel, same results) but takes its
 * scratch (per-row partial sums, status word, completion counter) from a fixed array inside the
 * library instead of a workspace.  It allocates nothing.
 *
 *   Arguments, layout and results are those of ce_with_grad, without workspace/workspace_bytes.
 *   B must not exceed FLCE_CE_NOALLOC_MAX_ROWS, else FLCE_ERR_UNSUPPORTED (flce_last_error() says
 *   why); use ce_with_grad with a workspace for larger batches.
 *   Memory: every GPU that loads the library holds the array (256 + 16 * FLCE_CE_NOALLOC_MAX_ROWS
 *   bytes, 4 MiB) until the process exits.
 *   The first call on each device looks up the array's device address (cudaGetSymbolAddress, with
 *   that device current) and remembers it; make that first call before any stream capture.  The remembered address belongs
 *   to the device's context of that moment: a caller that resets the device (cudaDeviceReset) or
 *   otherwise recreates its primary context must not call this entry point on that device again in
 *   the same process.
 *   All calls share the one array, which keeps the previous call's contents; each call clears what
 *   must start at zero.  Calls whose kernels can overlap on the GPU (e.g. on two streams without
 *   ordering between them, or from two host threads) race on the array: serialise them.
 *   The device status word cannot be read back through flce_read_device_status (there is no
 *   workspace); labels outside [0, V) are still treated as ignored rows.
 */
#define FLCE_CE_NOALLOC_MAX_ROWS 262144
flce_status ce_with_grad_noalloc(uint16_t* logits, const int64_t* labels, int64_t B, int64_t V,
                                 int64_t ignore_index, float z_loss, float* ce_sum, float* z_sum,
                                 int64_t* n_valid, void* stream);

/*
 * The reduced loss of the standalone CE from the device sums of ce_with_grad / ce_with_grad_ex, without
 * a host round trip (the loss a framework's autograd function returns):
 *   *loss = (*ce_sum + z_loss * *z_sum) / max(*n_valid, 1)   for FLCE_REDUCTION_MEAN ("Greyhound --
 *           Cross-Entropy", "Usage": ce_sum over the clamped valid count), or
 *   *loss = *ce_sum + z_loss * *z_sum                         for FLCE_REDUCTION_SUM.
 * With this z_loss the loss is the one whose gradient ce_with_grad writes (scaled by 1 / max(n_valid, 1)
 * for the mean).  All pointers are device pointers (n_valid 8-byte aligned, the others 4); one thread
 * of one kernel on `stream`.  FLCE_ERR_INVALID_ARG for a NULL pointer or another reduction.
 */
flce_status ce_reduce_loss(const float* ce_sum, const float* z_sum, const int64_t* n_valid, float z_loss,
                           int reduction, float* loss, void* stream);

/*
 * Multiplies a contiguous gradient buffer in place by an upstream gradient that lives on the device:
 *   grad[i] *= *upstream / (divisor != NULL ? max(*divisor, 1) : 1),   i in [0, n)
 * rounding to nearest-even in the buffer's type (dtype: FLCE_DTYPE_BF16, _F16 or _F32).  This is the
 * d_out factor of "Cut Cross Entropy visualized", "Breakdown: Backward Pass", step 4, applied after the
 * fact to gradients computed with an upstream gradient of 1 (flce_fwd_bwd, ce_with_grad): the backward
 * pass of an autograd function calls it with the incoming gradient, and for the standalone CE's mean
 * reduction with divisor = n_valid.  When the factor is exactly 1 the buffer is not touched.
 *   grad      device, 16-byte aligned (may be NULL when n == 0).
 *   upstream  [1] fp32, device.   divisor  [1] int64, device, or NULL.
 * FLCE_ERR_INVALID_ARG for a bad dtype, n < 0 or a NULL pointer; FLCE_ERR_MISALIGNED.
 */
flce_status flce_scale_gradient(void* grad, int dtype, int64_t n, const float* upstream, const int64_t* divisor,
                                void* stream);

/*
 * Copy the device status word of a workspace used by a previous call to *host_status, after
 * synchronising `stream`.  0 means no data error and no timeout.
 */
flce_status flce_read_device_status(const void* workspace, uint32_t* host_status, void* stream);

/* Human-readable name of a status code (static string). */
const char* flce_status_string(flce_status status);

/* Description of the last FLCE_ERR_CUDA / FLCE_ERR_UNSUPPORTED on this host thread (static buffer). */
const char* flce_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
