// gdn_graph.cu -- CUDA-graph decode buckets.
//
// A fixed decode graph per batch bucket (c1, c2, c4, ...) is how the Rocket
// post "A reduction barrier makes Qwen GDN graph replay bit exact" serves
// decode: immutable graphs over static buffers, inactive rows cleared on
// bucket transitions, slot 0 left untouched. Here one call captures one fused
// decode step (gdn_decode_step) over caller-owned buffers into an instantiated
// graph; replaying it costs one graph launch instead of argument checks and a
// kernel launch. A bucket serves fewer rows than its size by giving the unused
// rows slot 0: by the slot contract their outputs are written as zeros and no
// state is touched.
#include <new>

#include "gdn_internal.h"

struct gdn_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" {

gdn_status gdn_decode_graph_create(const void* mixed_qkv, const void* a, const void* b,
                                   gdn_gate_mode gate_mode, const float* A_log,
                                   const float* dt_bias, const void* conv_weight,
                                   const void* conv_bias, int32_t silu, void* conv_state,
                                   gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                                   float* ssm_state, const int32_t* slot, int32_t batch,
                                   int32_t num_slots, gdn_dims dims, float scale,
                                   int32_t qk_l2norm, const gdn_output_gate* gate, void* out,
                                   gdn_dtype out_dtype, int32_t* err, gdn_graph** graph_out) {
  if (!graph_out) return GDN_ERR_INVALID_ARG;
  *graph_out = nullptr;
  if (batch <= 0) return GDN_ERR_INVALID_ARG;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return GDN_ERR_CUDA;
  gdn_status st = GDN_OK;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return GDN_ERR_CUDA;
  }
  st = gdn_decode_step(mixed_qkv, a, b, gate_mode, A_log, dt_bias, conv_weight, conv_bias, silu,
                       conv_state, conv_dtype, conv_layout, ssm_state, slot, batch, num_slots,
                       dims, scale, qk_l2norm, gate, out, out_dtype, err, cs);
  const cudaError_t ce = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (st != GDN_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (ce != cudaSuccess || !g) return GDN_ERR_CUDA;
  gdn_graph* h = new (std::nothrow) gdn_graph;
  if (!h) {
    cudaGraphDestroy(g);
    return GDN_ERR_CUDA;
  }
  h->graph = g;
  if (cudaGraphInstantiate(&h->exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    delete h;
    return GDN_ERR_CUDA;
  }
  *graph_out = h;
  return GDN_OK;
}

gdn_status gdn_graph_launch(gdn_graph* graph, void* stream) {
  if (!graph || !graph->exec) return GDN_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GDN_OK
             : GDN_ERR_CUDA;
}

void gdn_graph_destroy(gdn_graph* graph) {
  if (!graph) return;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
}

}  // extern "C"
