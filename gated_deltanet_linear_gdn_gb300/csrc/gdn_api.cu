// gdn_api.cu -- the C ABI declared in include/gdn.h: argument checks, launch
// configuration and error mapping. No allocation, no synchronisation: every
// call only enqueues kernels on the caller's stream.
#include <algorithm>
#include <vector>

#include "gdn_internal.h"
#include "gdn_testing.h"

namespace {

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

gdn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

bool valid_dtype(gdn_dtype d) { return d == GDN_BF16 || d == GDN_F32; }
bool valid_layout(gdn_conv_layout l) { return l == GDN_CONV_DIM_FIRST || l == GDN_CONV_TAP_FIRST; }

// Shared checks of the layer calls. Returns GDN_OK and fills `la` when valid.
gdn_status check_layer(const void* mixed, const void* a, const void* b, gdn_gate_mode gate_mode,
                       const float* A_log, const float* dt_bias, const void* conv_w,
                       const void* conv_b, int32_t silu, void* conv_state, gdn_dtype conv_dtype,
                       gdn_conv_layout conv_layout, float* ssm, const int32_t* slot,
                       int32_t num_slots, gdn_dims d, float scale, int32_t qk_l2norm, void* out,
                       gdn_dtype out_dtype, int32_t* err, gdn::LayerArgs& la) {
  if (d.num_k_heads <= 0 || d.num_v_heads <= 0 || d.head_k_dim <= 0 || d.head_v_dim <= 0)
    return GDN_ERR_INVALID_ARG;
  if (d.num_v_heads % d.num_k_heads != 0) return GDN_ERR_INVALID_ARG;
  if (d.state_bf16 != 0 && d.state_bf16 != 1) return GDN_ERR_INVALID_ARG;
  if (num_slots < 1) return GDN_ERR_INVALID_ARG;
  if (gate_mode != GDN_GATE_FUSED && gate_mode != GDN_GATE_DIRECT) return GDN_ERR_INVALID_ARG;
  if (!valid_dtype(out_dtype)) return GDN_ERR_INVALID_ARG;
  if (!mixed || !a || !b || !ssm || !slot || !out) return GDN_ERR_INVALID_ARG;
  if (gate_mode == GDN_GATE_FUSED && (!A_log || !dt_bias)) return GDN_ERR_INVALID_ARG;
  if (conv_w) {
    if (!conv_state || !valid_dtype(conv_dtype) || !valid_layout(conv_layout))
      return GDN_ERR_INVALID_ARG;
    if (d.conv_width != gdn::kConvWidth) return GDN_ERR_UNSUPPORTED;
    if (!aligned(conv_w, 16) || !aligned(conv_state, 16) || (conv_b && !aligned(conv_b, 16)))
      return GDN_ERR_INVALID_ARG;
  }
  if (d.head_k_dim != d.head_v_dim) return GDN_ERR_UNSUPPORTED;
  if (d.head_k_dim != 32 && d.head_k_dim != 64 && d.head_k_dim != 128) return GDN_ERR_UNSUPPORTED;
  const int r = d.num_v_heads / d.num_k_heads;
  if (r != 1 && r != 2 && r != 4) return GDN_ERR_UNSUPPORTED;
  if (d.num_v_heads > 65535) return GDN_ERR_UNSUPPORTED;
  if (!aligned(mixed, 16) || !aligned(ssm, 16) || !aligned(out, 4) || !aligned(slot, 4) ||
      !aligned(a, 4) || !aligned(b, 4))
    return GDN_ERR_INVALID_ARG;
  la.mixed = mixed;
  la.a = a;
  la.b = b;
  la.gate_mode = gate_mode;
  la.A_log = A_log;
  la.dt_bias = dt_bias;
  la.conv_w = conv_w;
  la.conv_b = conv_w ? conv_b : nullptr;
  la.silu = silu != 0;
  la.conv_state = conv_state;
  la.conv_f32 = conv_dtype == GDN_F32;
  la.conv_layout = conv_layout;
  la.ssm = ssm;
  la.ssm_bf16 = d.state_bf16;
  la.slot = slot;
  la.num_slots = num_slots;
  la.Hk = d.num_k_heads;
  la.Hv = d.num_v_heads;
  la.dk = d.head_k_dim;
  la.dv = d.head_v_dim;
  la.D = 2 * d.num_k_heads * d.head_k_dim + d.num_v_heads * d.head_v_dim;
  la.scale = scale;
  la.qk_l2norm = qk_l2norm != 0;
  la.out = out;
  la.out_f32 = out_dtype == GDN_F32;
  la.err = err;
  la.max_ctas = 0;
  return GDN_OK;
}

// The optional output gate: NULL leaves `la` ungated.
gdn_status check_gate(const gdn_output_gate* g, gdn::LayerArgs& la) {
  la.gated = 0;
  la.gate_z = nullptr;
  la.gate_w = nullptr;
  la.gate_offset = 0.0f;
  la.gate_eps = 0.0f;
  la.gate_act = 0;
  if (!g) return GDN_OK;
  if (!g->z || !g->weight || !aligned(g->z, 16) || !aligned(g->weight, 16))
    return GDN_ERR_INVALID_ARG;
  if (g->act != GDN_ACT_SILU && g->act != GDN_ACT_SIGMOID) return GDN_ERR_INVALID_ARG;
  if (!(g->eps >= 0.0f) || !(g->eps < 3.0e38f) || !(g->weight_offset == g->weight_offset))
    return GDN_ERR_INVALID_ARG;  // eps finite and non-negative, offset not NaN
  la.gated = 1;
  la.gate_z = g->z;
  la.gate_w = g->weight;
  la.gate_offset = g->weight_offset;
  la.gate_eps = g->eps;
  la.gate_act = g->act;
  return GDN_OK;
}

}  // namespace

namespace gdn {

gdn_status prepare_decode(const void* mixed_qkv, const void* a, const void* b,
                          gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                          const void* conv_weight, const void* conv_bias, int32_t silu,
                          void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                          float* ssm_state, const int32_t* slot, int32_t batch, int32_t num_slots,
                          gdn_dims dims, float scale, int32_t qk_l2norm,
                          const gdn_output_gate* gate, void* out, gdn_dtype out_dtype,
                          int32_t* err, LayerArgs& la) {
  if (batch <= 0) return GDN_ERR_INVALID_ARG;
  if (batch > 65535) return GDN_ERR_UNSUPPORTED;
  gdn_status st = check_layer(mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias,
                              silu, conv_state, conv_dtype, conv_layout, ssm_state, slot, num_slots,
                              dims, scale, qk_l2norm, out, out_dtype, err, la);
  if (st != GDN_OK) return st;
  st = check_gate(gate, la);
  if (st != GDN_OK) return st;
  if (la.gated && !aligned(out, 16)) return GDN_ERR_INVALID_ARG;  // 16-byte gated stores
  return GDN_OK;
}

gdn_status prepare_prefill(const void* mixed_qkv, const void* a, const void* b,
                           gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                           const void* conv_weight, const void* conv_bias, int32_t silu,
                           void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                           float* ssm_state, const int32_t* cu_seqlens, const int32_t* slot,
                           const uint8_t* has_initial_state, int32_t num_seqs,
                           int32_t total_tokens, int32_t num_slots, gdn_dims dims, float scale,
                           int32_t qk_l2norm, int32_t chunk, const gdn_output_gate* gate,
                           void* out, gdn_dtype out_dtype, void* workspace,
                           size_t workspace_bytes, int32_t* err, LayerArgs& la,
                           PrefillExtra& p) {
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (chunk != 16 && chunk != 32 && chunk != 64) return GDN_ERR_UNSUPPORTED;
  if (num_seqs == 0) return GDN_ERR_INVALID_ARG;  // (an empty call is the callers' no-op)
  if (num_seqs > 65535) return GDN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_seqs) * dims.num_v_heads > 0x7fffffff) return GDN_ERR_UNSUPPORTED;
  if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
  if (total_tokens == 0) {
    // no token is read or written: empty per-token arrays may be null
    const void* ph = ssm_state;
    if (!mixed_qkv) mixed_qkv = ph;
    if (!a) a = ph;
    if (!b) b = ph;
    if (!out) out = const_cast<void*>(ph);
  }
  gdn_status st = check_layer(mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias,
                              silu, conv_state, conv_dtype, conv_layout, ssm_state, slot, num_slots,
                              dims, scale, qk_l2norm, out, out_dtype, err, la);
  if (st != GDN_OK) return st;
  st = check_gate(gate, la);
  if (st != GDN_OK) return st;
  if (la.gated && total_tokens > 0 && !aligned(out, 16)) return GDN_ERR_INVALID_ARG;
  // the tensor-core state pass (dk = dv = 128) writes a bf16 output in 16-byte pieces
  if (!la.out_f32 && dims.head_k_dim == 128 && dims.head_v_dim == 128 && total_tokens > 0 &&
      !aligned(out, 16))
    return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_chunked_prefill_workspace_size(total_tokens, num_seqs, dims, chunk);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return GDN_ERR_INVALID_ARG;
  p = PrefillExtra{cu_seqlens, has_initial_state, num_seqs, total_tokens, chunk, workspace,
                   workspace_bytes, nullptr};
  return GDN_OK;
}

}  // namespace gdn

extern "C" {

gdn_status gdn_conv_update(const void* x, void* conv_state, gdn_dtype state_dtype,
                           gdn_conv_layout conv_layout, const void* weight, const void* bias,
                           int32_t silu, const int32_t* slot, int32_t batch, int32_t dim,
                           int32_t width, int32_t num_slots, void* out, int32_t* err,
                           void* stream) {
  if (batch < 0 || dim <= 0 || num_slots < 1) return GDN_ERR_INVALID_ARG;
  if (!valid_dtype(state_dtype) || !valid_layout(conv_layout)) return GDN_ERR_INVALID_ARG;
  if (width != gdn::kConvWidth || dim % 8 != 0) return GDN_ERR_UNSUPPORTED;
  if (batch > 65535) return GDN_ERR_UNSUPPORTED;
  if (batch == 0) return GDN_OK;
  if (!x || !conv_state || !weight || !slot || !out) return GDN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(conv_state, 16) || !aligned(weight, 16) || !aligned(out, 16) ||
      (bias && !aligned(bias, 16)) || !aligned(slot, 4))
    return GDN_ERR_INVALID_ARG;
  gdn::ConvUpdateArgs a{x, conv_state, state_dtype == GDN_F32, conv_layout, weight, bias,
                        silu != 0, slot, batch, dim, num_slots, out, err};
  return from_cuda(gdn::launch_conv_update(a, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_decode_step(const void* mixed_qkv, const void* a, const void* b,
                           gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                           const void* conv_weight, const void* conv_bias, int32_t silu,
                           void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                           float* ssm_state, const int32_t* slot, int32_t batch,
                           int32_t num_slots, gdn_dims dims, float scale, int32_t qk_l2norm,
                           const gdn_output_gate* gate, void* out, gdn_dtype out_dtype,
                           int32_t* err, void* stream) {
  if (batch == 0) return GDN_OK;
  gdn::LayerArgs la;
  const gdn_status st = gdn::prepare_decode(
      mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias, silu, conv_state,
      conv_dtype, conv_layout, ssm_state, slot, batch, num_slots, dims, scale, qk_l2norm, gate,
      out, out_dtype, err, la);
  if (st != GDN_OK) return st;
  return from_cuda(gdn::launch_decode(la, batch, static_cast<cudaStream_t>(stream)));
}

size_t gdn_chunked_prefill_workspace_size(int32_t total_tokens, int32_t num_seqs, gdn_dims dims,
                                          int32_t chunk) {
  if (total_tokens < 0 || num_seqs < 0 || (chunk != 16 && chunk != 32 && chunk != 64)) return 0;
  if (dims.num_k_heads <= 0 || dims.num_v_heads <= 0 || dims.head_k_dim <= 0 || dims.head_v_dim <= 0)
    return 0;
  // the conv buffer is always reserved, so one size serves both conv modes
  return gdn::prefill_workspace_bytes(total_tokens, num_seqs, dims.num_k_heads, dims.num_v_heads,
                                      dims.head_k_dim, dims.head_v_dim, chunk, 1);
}

gdn_status gdn_chunked_prefill(const void* mixed_qkv, const void* a, const void* b,
                               gdn_gate_mode gate_mode, const float* A_log,
                               const float* dt_bias, const void* conv_weight,
                               const void* conv_bias, int32_t silu, void* conv_state,
                               gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                               float* ssm_state, const int32_t* cu_seqlens, const int32_t* slot,
                               const uint8_t* has_initial_state, int32_t num_seqs,
                               int32_t total_tokens, int32_t num_slots, gdn_dims dims,
                               float scale, int32_t qk_l2norm, int32_t chunk,
                               const gdn_output_gate* gate, void* out, gdn_dtype out_dtype,
                               void* workspace, size_t workspace_bytes, int32_t* err,
                               void* stream) {
  if (num_seqs == 0 && total_tokens == 0 && (chunk == 16 || chunk == 32 || chunk == 64))
    return GDN_OK;
  gdn::LayerArgs la;
  gdn::PrefillExtra p;
  const gdn_status st = gdn::prepare_prefill(
      mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias, silu, conv_state,
      conv_dtype, conv_layout, ssm_state, cu_seqlens, slot, has_initial_state, num_seqs,
      total_tokens, num_slots, dims, scale, qk_l2norm, chunk, gate, out, out_dtype, workspace,
      workspace_bytes, err, la, p);
  if (st != GDN_OK) return st;
  return from_cuda(gdn::launch_prefill(la, p, static_cast<cudaStream_t>(stream)));
}

int32_t gdn_validate_slots(const int32_t* host_slot, int32_t n, int32_t num_slots) {
  if (n <= 0) return 0;
  if (!host_slot) return 1;
  std::vector<int32_t> active;
  active.reserve(n);
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = host_slot[i];
    if (s <= 0) continue;
    if (s >= num_slots) return 1;
    active.push_back(s);
  }
  std::sort(active.begin(), active.end());
  for (size_t i = 1; i < active.size(); ++i)
    if (active[i] == active[i - 1]) return 2;
  return 0;
}

gdn_status gdn_testing_set_fault(int32_t mode) {
  if (mode != GDN_TEST_FAULT_NONE && mode != GDN_TEST_FAULT_DECODE_CONSUMER &&
      mode != GDN_TEST_FAULT_PREFILL_PASS)
    return GDN_ERR_INVALID_ARG;
  const int d = mode == GDN_TEST_FAULT_DECODE_CONSUMER ? 1 : 0;
  const int p = mode == GDN_TEST_FAULT_PREFILL_PASS ? 2 : 0;
  if (gdn::set_decode_test_fault(d) != cudaSuccess) return GDN_ERR_CUDA;
  if (gdn::set_prefill_test_fault(p) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

const char* gdn_status_string(gdn_status status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null pointer, bad size or misaligned buffer";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: no kernel for this shape";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: kernel launch failed";
    case GDN_ERR_SCRATCH_LIMIT:
      return "GDN_ERR_SCRATCH_LIMIT: the call needs more than the library's fixed scratch "
             "(GDN_NOALLOC_SCRATCH_BYTES); use gdn_chunked_prefill with a workspace";
    default: return "unknown gdn_status";
  }
}

}  // extern "C"
