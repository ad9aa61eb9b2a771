// gdn_mixed.cu -- one call for a step that holds decode rows and prefill
// sequences together.
//
// The RL-Kernel PR #469 page ("C6: GDN decode-step goldens and recurrent/conv
// state contract", section "Not reproducible from this branch: the mixed
// decode+prefill measurement") reports that when a step also holds a prefill,
// the serving stack routes its decode rows through a different recurrent
// kernel, so their outputs and states depend on the step's composition; its
// cited fix routes mixed-step decodes through the packed decode kernel too.
// Here a mixed step runs its decode rows through the same fused decode kernel
// and its prefill sequences through the same chunked path as the separate
// calls, so every result is bitwise the separate calls' whatever the mix.
//
// Scheduling: the chunked prefill's state pass occupies one CTA per (sequence,
// value head) -- 32 of the 152 SMs for one Qwen3-Next sequence -- for most of
// its time. The decode rows are therefore enqueued on a side stream that waits
// for an event recorded just before that pass (before its last piece, when the
// prefill runs in pieces: no intra kernel runs beside it), with the decode grid
// capped to the SMs the pass leaves free; the caller's stream then waits for
// the side stream. The side stream and its two events are created once per device, on
// the first mixed call that needs them (make that call before any stream
// capture); mixed calls on one device enqueue one at a time.
#include <mutex>

#include "gdn_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t before_pass = nullptr;
  cudaEvent_t done = nullptr;
};
SideStream g_side[kMaxDevices];

// The current device's side stream, created on first use. The caller holds g_mu.
cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStream& s = g_side[dev];
  if (!s.stream) {
    if ((e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.before_pass, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  *out = &s;
  return cudaSuccess;
}

size_t elem(gdn_dtype d) { return d == GDN_F32 ? 4 : 2; }

const void* offset(const void* p, size_t bytes) {
  return p ? static_cast<const char*>(p) + bytes : nullptr;
}

}  // namespace

extern "C" gdn_status gdn_mixed_step(
    const void* mixed_qkv, const void* a, const void* b, gdn_gate_mode gate_mode,
    const float* A_log, const float* dt_bias, const void* conv_weight, const void* conv_bias,
    int32_t silu, void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
    float* ssm_state, const int32_t* slot, int32_t num_decode, const int32_t* cu_seqlens,
    const uint8_t* has_initial_state, int32_t num_prefill_seqs, int32_t prefill_tokens,
    int32_t num_slots, gdn_dims dims, float scale, int32_t qk_l2norm, int32_t chunk,
    const gdn_output_gate* gate, void* out, gdn_dtype out_dtype, void* workspace,
    size_t workspace_bytes, int32_t* err, void* stream) {
  if (num_decode < 0 || num_prefill_seqs < 0 || prefill_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (num_prefill_seqs == 0 && prefill_tokens != 0) return GDN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool dec = num_decode > 0, pre = num_prefill_seqs > 0;
  gdn::LayerArgs ld, lp;
  gdn::PrefillExtra p;
  if (dec) {
    const gdn_status st = gdn::prepare_decode(
        mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias, silu, conv_state,
        conv_dtype, conv_layout, ssm_state, slot, num_decode, num_slots, dims, scale, qk_l2norm,
        gate, out, out_dtype, err, ld);
    if (st != GDN_OK) return st;
  }
  if (pre) {
    // the prefill part starts num_decode token rows (and slots) in
    const size_t rows = static_cast<size_t>(num_decode);
    const int D = 2 * dims.num_k_heads * dims.head_k_dim + dims.num_v_heads * dims.head_v_dim;
    const size_t ab = gate_mode == GDN_GATE_DIRECT ? 4 : 2;
    const size_t hv = static_cast<size_t>(dims.num_v_heads), dv = static_cast<size_t>(dims.head_v_dim);
    gdn_output_gate gp;
    const gdn_output_gate* gpp = nullptr;
    if (gate) {
      gp = *gate;
      gp.z = offset(gate->z, rows * hv * dv * 2);
      gpp = &gp;
    }
    const gdn_status st = gdn::prepare_prefill(
        offset(mixed_qkv, rows * D * 2), offset(a, rows * hv * ab), offset(b, rows * hv * ab),
        gate_mode, A_log, dt_bias, conv_weight, conv_bias, silu, conv_state, conv_dtype,
        conv_layout, ssm_state, cu_seqlens, slot ? slot + num_decode : nullptr, has_initial_state,
        num_prefill_seqs, prefill_tokens, num_slots, dims, scale, qk_l2norm, chunk, gpp,
        const_cast<void*>(offset(out, rows * hv * dv * elem(out_dtype))), out_dtype, workspace,
        workspace_bytes, err, lp, p);
    if (st != GDN_OK) return st;
  }
  if (!dec && !pre) return GDN_OK;
  if (!pre) return gdn::launch_decode(ld, num_decode, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
  if (!dec) return gdn::launch_prefill(lp, p, s) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;

  // One mixed enqueue at a time: the event record, the side stream's wait on it
  // and the decode launch must not interleave with another call's.
  std::lock_guard<std::mutex> lock(g_mu);
  SideStream* side = nullptr;
  if (side_stream(&side) != cudaSuccess) return GDN_ERR_CUDA;
  p.before_pass = side->before_pass;
  // the decode grid takes the SMs that the state pass leaves free
  const int sms = gdn::sm_count();
  const int pass_ctas = num_prefill_seqs * dims.num_v_heads *
                        (dims.head_k_dim == 128 && dims.head_v_dim == 128 ? 1 : 2);
  ld.max_ctas = pass_ctas < sms - 16 ? sms - pass_ctas : 0;
  if (gdn::launch_prefill(lp, p, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamWaitEvent(side->stream, side->before_pass, 0) != cudaSuccess) return GDN_ERR_CUDA;
  if (gdn::launch_decode(ld, num_decode, side->stream) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaEventRecord(side->done, side->stream) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamWaitEvent(s, side->done, 0) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}
