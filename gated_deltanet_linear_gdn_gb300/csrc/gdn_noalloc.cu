// gdn_noalloc.cu -- chunked prefill for callers that cannot allocate device
// memory.
//
// gdn_chunked_prefill needs a caller-provided workspace. Some callers cannot
// provide one: code running where no allocator may be called (a host thread
// that must not synchronise, which cudaMalloc can do; an embedding runtime
// that owns every device allocation and exposes none to plug-ins; a process
// that has to keep a fixed memory footprint after start-up). For them this file
// keeps the workspace in a fixed-size array in the library's own device
// memory, declared below, and calls the ordinary prefill path with it.
//
// Costs and limits (also stated in include/gdn.h):
//  - every GPU on which the library is loaded holds GDN_NOALLOC_SCRATCH_BYTES of
//    device memory for this array until the process exits;
//  - requests whose workspace would exceed that size are rejected with
//    GDN_ERR_SCRATCH_LIMIT before anything is enqueued;
//  - all calls on one device share the one array, so calls that can overlap on
//    the GPU (different streams without ordering between them) race on it;
//  - the first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (which may load the module), so make that first call
//    before any stream capture.
// The prefill writes every scratch word before it reads it, so the array keeps
// whatever the previous call left and is never cleared.
#include <mutex>

#include "gdn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_prefill_scratch on the current device (looked up once per
// device; the host-side symbol itself is only a stand-in and must never be
// passed to a kernel).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" gdn_status gdn_chunked_prefill_noalloc(
    const void* mixed_qkv, const void* a, const void* b, gdn_gate_mode gate_mode,
    const float* A_log, const float* dt_bias, const void* conv_weight, const void* conv_bias,
    int32_t silu, void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
    float* ssm_state, const int32_t* cu_seqlens, const int32_t* slot,
    const uint8_t* has_initial_state, int32_t num_seqs, int32_t total_tokens, int32_t num_slots,
    gdn_dims dims, float scale, int32_t qk_l2norm, int32_t chunk, const gdn_output_gate* gate,
    void* out, gdn_dtype out_dtype, int32_t* err, void* stream) {
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_chunked_prefill_workspace_size(total_tokens, num_seqs, dims, chunk);
  if (need == 0) {
    // sizes the ordinary entry point rejects: let it report the same status
    return gdn_chunked_prefill(mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight,
                               conv_bias, silu, conv_state, conv_dtype, conv_layout, ssm_state,
                               cu_seqlens, slot, has_initial_state, num_seqs, total_tokens,
                               num_slots, dims, scale, qk_l2norm, chunk, gate, out, out_dtype,
                               nullptr, 0, err, stream);
  }
  if (need > static_cast<size_t>(GDN_NOALLOC_SCRATCH_BYTES)) return GDN_ERR_SCRATCH_LIMIT;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return GDN_ERR_CUDA;
  return gdn_chunked_prefill(mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias,
                             silu, conv_state, conv_dtype, conv_layout, ssm_state, cu_seqlens,
                             slot, has_initial_state, num_seqs, total_tokens, num_slots, dims,
                             scale, qk_l2norm, chunk, gate, out, out_dtype, ws,
                             static_cast<size_t>(GDN_NOALLOC_SCRATCH_BYTES), err, stream);
}
