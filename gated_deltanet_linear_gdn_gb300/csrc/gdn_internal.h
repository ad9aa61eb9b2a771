// gdn_internal.h -- launcher declarations shared between the C-ABI layer and
// the kernel translation units. Host-only types; no torch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kConvWidth = 4;  // the only conv width with kernels

struct ConvUpdateArgs {
  const void* x;
  void* conv_state;
  int f32_cache;
  int layout;
  const void* weight;
  const void* bias;
  int silu;
  const int32_t* slot;
  int B, D, num_slots;
  void* out;
  int32_t* err;
};

struct LayerArgs {
  const void* mixed;  // [T, D] bf16
  const void* a;
  const void* b;
  int gate_mode;
  const float* A_log;
  const float* dt_bias;
  const void* conv_w;  // null = conv bypass
  const void* conv_b;
  int silu;
  void* conv_state;
  int conv_f32;
  int conv_layout;
  float* ssm;  // [num_slots, Hv, dv, dk], fp32 or (ssm_bf16) bf16 data
  int ssm_bf16;
  const int32_t* slot;
  int num_slots;
  int Hk, Hv, dk, dv, D;
  float scale;
  int qk_l2norm;
  void* out;
  int out_f32;
  int32_t* err;
  // output gate (gated RMSNorm of o per value head); gated == 0: out = o
  int gated;
  const void* gate_z;  // [tokens, Hv, dv] bf16
  const float* gate_w; // [dv]
  float gate_offset;
  float gate_eps;
  int gate_act;        // gdn_gate_act
  int max_ctas;        // decode: cap on the persistent grid (0 = one CTA per SM)
};

struct PrefillExtra {
  const int32_t* cu_seqlens;
  const uint8_t* has_init;
  int num_seqs;
  int total_tokens;
  int chunk;
  void* workspace;
  size_t workspace_bytes;
  cudaEvent_t before_pass;  // recorded on the stream just before the (last) state pass (nullable)
};

cudaError_t launch_conv_update(const ConvUpdateArgs& a, cudaStream_t s);

// Argument checks of the decode and prefill calls (gdn_api.cu), without launching:
// on GDN_OK `la` (and `p`) describe the call.
gdn_status prepare_decode(const void* mixed_qkv, const void* a, const void* b,
                          gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                          const void* conv_weight, const void* conv_bias, int32_t silu,
                          void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                          float* ssm_state, const int32_t* slot, int32_t batch, int32_t num_slots,
                          gdn_dims dims, float scale, int32_t qk_l2norm,
                          const gdn_output_gate* gate, void* out, gdn_dtype out_dtype,
                          int32_t* err, LayerArgs& la);
gdn_status prepare_prefill(const void* mixed_qkv, const void* a, const void* b,
                           gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                           const void* conv_weight, const void* conv_bias, int32_t silu,
                           void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                           float* ssm_state, const int32_t* cu_seqlens, const int32_t* slot,
                           const uint8_t* has_initial_state, int32_t num_seqs,
                           int32_t total_tokens, int32_t num_slots, gdn_dims dims, float scale,
                           int32_t qk_l2norm, int32_t chunk, const gdn_output_gate* gate,
                           void* out, gdn_dtype out_dtype, void* workspace,
                           size_t workspace_bytes, int32_t* err, LayerArgs& la, PrefillExtra& p);
int sm_count();  // SMs of the current device (gdn_decode.cu)
cudaError_t launch_decode(const LayerArgs& a, int B, cudaStream_t s);
// the output gate in place over `rows` rows of dv values of a.out (gdn_gate.cu)
cudaError_t launch_output_gate(const LayerArgs& a, int64_t rows, cudaStream_t s);
cudaError_t launch_prefill(const LayerArgs& a, const PrefillExtra& p, cudaStream_t s);
size_t prefill_workspace_bytes(int total_tokens, int num_seqs, int Hk, int Hv, int dk, int dv,
                               int chunk, int conv);

// chunk table + sequence checks (gdn_prefill.cu): meta[0] = number of chunks,
// seq_ok[i], chunk_off[N+1] (first chunk of each sequence), chunk_seq[chunk], and (when
// seq_order is not null) seq_order[N], the sequences by descending chunk count
cudaError_t launch_prefill_prep(const LayerArgs& a, const PrefillExtra& p, int32_t* meta,
                                int32_t* seq_ok, int32_t* chunk_off, int32_t* chunk_seq,
                                int32_t* seq_order, cudaStream_t s);
// tensor-core path for dk = dv = 128 (gdn_prefill_tc.cu)
size_t prefill_tc_workspace_bytes(int total_tokens, int num_seqs, int Hk, int Hv, int chunk);
cudaError_t launch_prefill_tc(const LayerArgs& a, const PrefillExtra& p, cudaStream_t s);

// test hooks (gdn_testing_set_fault): the device flag of the decode and of the tensor-core
// prefill translation units
cudaError_t set_decode_test_fault(int mode);
cudaError_t set_prefill_test_fault(int mode);

// prefill helpers implemented in gdn_conv.cu: the conv output y of every token of an active
// sequence (over the chunk table of launch_prefill_prep), then each active sequence's final
// conv window
cudaError_t launch_prefill_conv(const LayerArgs& a, const PrefillExtra& p, const int32_t* meta,
                                const int32_t* seq_ok, const int32_t* chunk_off,
                                const int32_t* chunk_seq, int max_chunks, uint16_t* y,
                                cudaStream_t s);

}  // namespace gdn
