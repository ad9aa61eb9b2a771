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
//  - the first call under each CUDA context looks up the array's device address
//    with cudaGetSymbolAddress (which may load the module), so make that first
//    call before any stream capture. The address is kept per context; a context
//    destroyed and recreated under the same handle (cudaDeviceReset on the
//    primary context) is not detected, so a caller that resets the device does
//    not use this entry point afterwards.
// Arguments are checked in full before the look-up: a bad call returns its
// status without touching the CUDA runtime.
// The prefill writes every scratch word before it reads it, so the array keeps
// whatever the previous call left and is never cleared.
#include <mutex>

#include "gdn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_NOALLOC_SCRATCH_BYTES];

// cuCtxGetCurrent, fetched through the runtime (so the library links no driver library)
typedef int (*CtxGetCurrentFn)(void** ctx);

constexpr int kMaxContexts = 64;
struct ScratchEntry {
  void* ctx;
  void* ptr;
};
std::mutex g_mu;
ScratchEntry g_table[kMaxContexts] = {};
int g_used = 0;
CtxGetCurrentFn g_ctx_get = nullptr;
bool g_ctx_get_tried = false;

// The current context's handle, or null if it cannot be had (then nothing is cached).
void* current_context() {
  if (!g_ctx_get_tried) {
    g_ctx_get_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  void* ctx = nullptr;
  if (!g_ctx_get || g_ctx_get(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of g_prefill_scratch in the current context (looked up once per context;
// the host-side symbol itself is only a stand-in and must never be passed to a kernel).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);  // makes the device's primary context current if none is
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  void* ctx = current_context();
  if (ctx) {
    for (int i = 0; i < g_used; ++i)
      if (g_table[i].ctx == ctx) {
        *out = g_table[i].ptr;
        return cudaSuccess;
      }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_prefill_scratch);
  if (e != cudaSuccess) return e;
  if (ctx && g_used < kMaxContexts) g_table[g_used++] = ScratchEntry{ctx, p};
  *out = p;
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
  if (num_seqs == 0 && total_tokens == 0 && (chunk == 16 || chunk == 32 || chunk == 64))
    return GDN_OK;  // the ordinary entry point's no-op
  const size_t need = gdn_chunked_prefill_workspace_size(total_tokens, num_seqs, dims, chunk);
  if (need > static_cast<size_t>(GDN_NOALLOC_SCRATCH_BYTES)) return GDN_ERR_SCRATCH_LIMIT;
  // every argument check of the ordinary entry point, with a stand-in workspace of the
  // scratch's size (an aligned non-null value that is never dereferenced)
  gdn::LayerArgs la;
  gdn::PrefillExtra p;
  const gdn_status st = gdn::prepare_prefill(
      mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias, silu, conv_state,
      conv_dtype, conv_layout, ssm_state, cu_seqlens, slot, has_initial_state, num_seqs,
      total_tokens, num_slots, dims, scale, qk_l2norm, chunk, gate, out, out_dtype,
      reinterpret_cast<void*>(static_cast<uintptr_t>(256)),
      static_cast<size_t>(GDN_NOALLOC_SCRATCH_BYTES), err, la, p);
  if (st != GDN_OK) return st;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return GDN_ERR_CUDA;
  p.workspace = ws;
  return gdn::launch_prefill(la, p, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}
