// flce_launch.cu -- enqueues every pass of one flce_fwd_bwd call on the caller's stream, no host
// synchronisation, no allocation, optional caller events at the pass boundaries:
//   header clear -> [vocabulary sort (vocab_sort.cu)] -> then either
//   online flow (grad_input requested):
//     bias table + valid count -> grad_input pass that also finds the LSE (flce_bwd.cu, online form)
//     -> loss reduction -> [LSE tiles, merge, reduction, classic grad_input pass: gated, they run only when
//     the online pass reported a row outside its safe range] -> grad_W / grad_bias pass
//   or classic flow:
//     LSE tiles (flce_fwd.cu) -> split merge -> loss reduction -> grad_input and grad_W passes (one launch
//     when both run)
#include "flce_kernels.cuh"

namespace flce {

cudaError_t launch_lse_passes(const FusedArgs& a, const FusedWorkspace& ws, int num_sms, cudaStream_t stream,
                              char* err, size_t err_len, cudaEvent_t const* events, const uint32_t* gate);
cudaError_t launch_online_prep(const FusedArgs& a, const FusedWorkspace& ws, cudaStream_t stream);
cudaError_t launch_loss_reduce(const FusedArgs& a, const FusedWorkspace& ws, cudaStream_t stream);

cudaError_t launch_fused(const FusedArgs& args, void* workspace, int num_sms, cudaStream_t stream, char* err,
                         size_t err_len, cudaEvent_t const* events) {
  const FusedWorkspace ws = carve_workspace(workspace, args.BT, args.V);
  auto mark = [&](int i) { return events != nullptr ? cudaEventRecord(events[i], stream) : cudaSuccess; };
  cudaError_t e = cudaMemsetAsync(workspace, 0, 256, stream);
  if (e != cudaSuccess) return e;
  if ((e = mark(0)) != cudaSuccess) return e;
  FusedArgs a = args;
  const int32_t* row_perm = nullptr;
  if (args.sort_vocab) {
    // every pass below runs on the sorted vocabulary (sorted W, bias and targets, ignore index -1); the
    // grad_W pass maps its rows back to the caller's order
    const VocabSortWorkspace vs = carve_vocab_sort(
        static_cast<unsigned char*>(workspace) + fused_workspace_bytes(args.BT, args.V), args.BT, args.H, args.V);
    if ((e = launch_vocab_sort(args, vs, ws.status, num_sms, stream)) != cudaSuccess) return e;
    const size_t vb = sizeof(float) * static_cast<size_t>(args.V);
    if (args.logit_avg_out != nullptr &&
        (e = cudaMemcpyAsync(args.logit_avg_out, vs.logit_avg, vb, cudaMemcpyDeviceToDevice, stream)) != cudaSuccess)
      return e;
    if (args.vocab_order_out != nullptr &&
        (e = cudaMemcpyAsync(args.vocab_order_out, vs.vals[0], vb, cudaMemcpyDeviceToDevice, stream)) != cudaSuccess)
      return e;
    a.W = vs.W;
    a.bias = args.bias != nullptr ? vs.bias : nullptr;
    a.target = vs.target;
    a.ignore_index = -1;
    row_perm = vs.vals[0];
  }
  const bool want_dw = (a.grad_W != nullptr) || (a.grad_bias != nullptr);
  // (with gradient filtering the online grad_input pass is exact and only the grad_W pass filters)
  const bool online = a.BT > 0 && a.grad_input != nullptr && !a.separate_lse;
  DgPairArgs pa{};
  pa.bias = a.bias;
  pa.stats = ws.stats;
  pa.stats_ct = ws.stats_ct;
  pa.colb2 = ws.colb2;
  pa.scale = ws.scale;
  pa.zf_neg = ws.zf_neg;
  pa.z_loss = a.z_loss;
  pa.accumulate = a.accumulate;
  pa.filter_eps = a.filter_eps;
  pa.skip_count = ws.skipped;
  pa.row_perm = row_perm;
  pa.BT = static_cast<int>(a.BT);
  pa.V = static_cast<int>(a.V);
  pa.H = static_cast<int>(a.H);
  pa.grad_input = a.grad_input;
  pa.grad_W = a.grad_W;
  pa.grad_bias = a.grad_bias;
  pa.status = ws.status;
  // (read by the grad_W pass only)
  pa.token_splits = a.token_splits;
  pa.debug_stall_us = a.debug_stall_us;
  pa.split_scratch = reinterpret_cast<float*>(ws.part);
  pa.split_scratch_bytes = ws.part_bytes;
  pa.split_count = ws.ts_count;
  pa.work_q = ws.work_q + 1;     // (the grad_W pass; the gated classic grad_input pass takes none)
  pa.side_count = ws.side_count;
  pa.single_count = ws.single_count;
  pa.single_units = ws.single_units + 1;
  if (online) {
    // events: 1 after the bias table and count, 2 after the online grad_input pass, 3 after the loss
    // reduction and the gated classic passes, 4 after the grad_W pass
    if ((e = launch_online_prep(a, ws, stream)) != cudaSuccess) return e;
    if ((e = mark(1)) != cudaSuccess) return e;
    CUtensorMap tm_h, tm_w;
    if (!make_tmap_bf16(&tm_h, a.hidden, a.BT, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tm_w, a.W, a.V, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
    DgPairArgs po = pa;
    po.target = a.target;
    po.ignore_index = a.ignore_index;
    po.grad_tok = a.grad_tok;
    po.Wmat = a.W;
    po.mref_g = ws.part_t;                      // the split partials are free in this flow
    po.part_g = reinterpret_cast<float4*>(ws.part);   // [BT up to 256][4][2] float4 fits its 32 x BTp float2
    po.entropy_out = a.entropy;
    po.row_redo = ws.row_redo;
    po.stats_out = ws.stats;
    po.stats_ct_out = ws.stats_ct;
    po.row_loss = ws.row_loss;
    po.loss_tok = a.loss_tok;
    po.zf_neg_out = ws.zf_neg;
    po.fallback = ws.fallback;
    po.vocab_splits = a.vocab_splits;
    po.vs_mref = ws.vs_mref;
    po.vs_part = ws.vs_part;
    po.vs_stat = ws.vs_stat;
    po.vs_o = ws.split_acc;
    po.vs_count = ws.vs_count;
    po.work_q = ws.work_q;
    po.single_units = ws.single_units;
    if ((e = launch_dgrad_online(tm_h, tm_w, po, stream)) != cudaSuccess) return e;
    if ((e = mark(2)) != cudaSuccess) return e;
    if ((e = launch_loss_reduce(a, ws, stream)) != cudaSuccess) return e;
    // the classic passes, run only if the online pass set the fallback flag
    if ((e = launch_lse_passes(a, ws, num_sms, stream, err, err_len, nullptr, ws.fallback)) != cudaSuccess) return e;
    DgPairArgs pg = pa;
    pg.gate = ws.fallback;
    pg.work_q = nullptr;
    pg.row_redo = ws.row_redo;   // only the rows the online pass left
    if ((e = launch_dgrad_pair<false>(tm_h, tm_w, pg, stream)) != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    if (want_dw && (e = launch_dgrad_pair<true>(tm_w, tm_h, pa, stream)) != cudaSuccess) return e;
    return mark(4);
  }
  if ((e = launch_lse_passes(a, ws, num_sms, stream, err, err_len, events, nullptr)) != cudaSuccess) return e;
  if ((e = mark(2)) != cudaSuccess) return e;

  if (a.BT == 0) {
    // no tokens: every gradient is zero (unchanged when accumulating)
    if (!a.accumulate && a.grad_W != nullptr &&
        (e = cudaMemsetAsync(a.grad_W, 0, sizeof(float) * a.V * a.H, stream)) != cudaSuccess)
      return e;
    if (!a.accumulate && a.grad_bias != nullptr &&
        (e = cudaMemsetAsync(a.grad_bias, 0, sizeof(float) * a.V, stream)) != cudaSuccess)
      return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    return mark(4);
  }
  CUtensorMap tm_h128, tm_w128;
  if (a.grad_input != nullptr || want_dw) {
    if (!make_tmap_bf16(&tm_h128, a.hidden, a.BT, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tm_w128, a.W, a.V, a.H, kTileM, err, err_len)) return cudaErrorInvalidValue;
  }
  if (a.grad_input != nullptr && want_dw) {
    // both passes in one launch; caller events 3 and 4 are both recorded after it
    if ((e = launch_dgrad_both(tm_h128, tm_w128, pa, stream)) != cudaSuccess) return e;
    if ((e = mark(3)) != cudaSuccess) return e;
    return mark(4);
  }
  if (a.grad_input != nullptr) {
    DgPairArgs pi = pa;
    pi.work_q = ws.work_q;   // each pass has its own queue word (and count of single-pair units)
    pi.single_units = ws.single_units;
    if ((e = launch_dgrad_pair<false>(tm_h128, tm_w128, pi, stream)) != cudaSuccess) return e;
  }
  if ((e = mark(3)) != cudaSuccess) return e;
  if (want_dw) {
    if ((e = launch_dgrad_pair<true>(tm_w128, tm_h128, pa, stream)) != cudaSuccess) return e;
  }
  return mark(4);
}

}  // namespace flce
