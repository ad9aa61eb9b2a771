/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) layer hot path for GB300 (sm_103a).
 *
 * The library computes, on one GPU, the two halves of a GDN linear-attention
 * layer between its input and output projections:
 *
 *   1. the width-W causal depthwise conv1d (optionally followed by SiLU) over
 *      the packed q|k|v channels, which rolls a per-slot conv state, and
 *   2. the gated delta rule per value head h (k-head h / (Hv/Hk)):
 *        S <- a S ;  d = b (v - S k) ;  S <- S + d k^T ;  o = S q
 *      with a = exp(g), b = sigmoid(.), q and k L2-normalised, and an fp32
 *      state S of shape [dv, dk] addressed through a cache-slot table.
 *
 * Sources (by page title and section):
 *   [P1] RL-Kernel PR #469 "C6: GDN decode-step goldens and recurrent/conv
 *        state contract": Summary (state ABI, gating, QK norm, head mapping,
 *        conv accumulation) and Notes ("State ABI: index validation and the
 *        two NULL_BLOCK_ID contracts", "The conv half: coverage and the two
 *        mismatch mechanisms", "How the golden relates to the kernel").
 *   [P4] vLLM PR #53864 (CuteDSL GDN prefill, fourth Newton-Schulz round):
 *        "Numerical root cause and fix" -- the chunked prefill with a
 *        lower-triangular inverse of the per-chunk KK^T block.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless its comment says
 *     otherwise. The caller owns and allocates every buffer; the library never
 *     allocates, frees or synchronises inside these calls. Work is enqueued on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - All arrays are dense and row-major (C order) with the shapes given.
 *   - bf16 is IEEE bfloat16 bits (uint16); f32 is IEEE binary32.
 *   - Packed channels: D = 2*Hk*dk + Hv*dv, ordered [q (Hk*dk) | k (Hk*dk) |
 *     v (Hv*dv)], head-major inside each block ([P1] Summary: packed q/k/v).
 *   - Slot table ([P1] Notes, "State ABI"): slot <= 0 marks an inactive row or
 *     sequence: its outputs are written as zeros and no state is touched.
 *     slot >= num_slots sets GDN_DEVERR_SLOT_RANGE in *err (when err != NULL)
 *     and the row is treated as inactive. Repeated active slots are NOT
 *     detected on the device (two rows would race on one state block); use
 *     gdn_validate_slots on the host where that matters.
 *   - Errors: argument errors return before any launch and leave every buffer
 *     untouched. A failed launch returns GDN_ERR_CUDA. Nothing traps.
 *   - Results are deterministic: no atomic arithmetic (atomics only set bits of
 *     the error word), no batch-dependent reduction order; each row / sequence
 *     depends only on its own inputs and slot.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* a null pointer, a bad size or an inconsistent shape */
  GDN_ERR_UNSUPPORTED = 2, /* a valid shape this build has no kernel for */
  GDN_ERR_CUDA = 3,        /* the launch failed (cudaGetLastError != success) */
  GDN_ERR_SCRATCH_LIMIT = 4 /* gdn_chunked_prefill_noalloc: the call needs more scratch
                               than GDN_NOALLOC_SCRATCH_BYTES */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/* Conv state pool layout.  DIM_FIRST: [num_slots, D, W-1];  TAP_FIRST:
 * [num_slots, W-1, D].  Tap 0 is the oldest cached input in both. */
typedef enum { GDN_CONV_DIM_FIRST = 0, GDN_CONV_TAP_FIRST = 1 } gdn_conv_layout;

/* FUSED: a, b are bf16 [rows, Hv] projections; g = -exp(A_log) * softplus(a +
 *        dt_bias) (softplus(x) = x for x > 20) and beta = sigmoid(b), in fp32
 *        ([P1] Notes, "How the golden relates to the kernel", item 1).
 * DIRECT: a holds g and b holds beta, both f32 [rows, Hv]; A_log and dt_bias
 *        are ignored and may be NULL. */
typedef enum { GDN_GATE_FUSED = 0, GDN_GATE_DIRECT = 1 } gdn_gate_mode;

typedef struct {
  int32_t num_k_heads; /* Hk */
  int32_t num_v_heads; /* Hv (a multiple of Hk) */
  int32_t head_k_dim;  /* dk */
  int32_t head_v_dim;  /* dv */
  int32_t conv_width;  /* W */
  /* Recurrent-state storage: 0 = fp32 (default), 1 = bf16. The arithmetic stays fp32;
   * only the write into the pool rounds to bf16 (round to nearest even), as the state
   * ABI of RL-Kernel PR #469 "C6: GDN decode-step goldens and recurrent/conv state
   * contract" (Summary) has it. With 1, `ssm_state` points at bf16 data of the same
   * shape. */
  int32_t state_bf16;
} gdn_dims;

/*
 * Output gate of the GDN block: a gated RMSNorm of the core output o over each
 * value head, before the output projection ([P1] Summary by CodeRabbit -- SiLU
 * or sigmoid gating -- and Walkthrough -- a weight offset -- on the stacked
 * gated-RMSNorm PRs #466-#468). Per token t and value
 * head h, with o the core output:
 *   out[t, h, i] = o[i] / sqrt(mean_j o[j]^2 + eps) * (weight[i] + weight_offset)
 *                  * act(z[t, h, i]),   act = SiLU (z * sigmoid(z)) or sigmoid,
 * and an all-zero o with eps 0 gating to zero. The norm comes before the gate.
 * Arithmetic is fp32; the result is stored in out_dtype. The decode step gates
 * the unrounded fp32 o inside its own kernel; the chunked prefill stores o in
 * out_dtype first and gates it in place after its state pass (with a bf16
 * output that is the block's unfused arithmetic). weight_offset is 0 for the
 * plain form and 1 for the zero-centred one (weight stored as w - 1). `out`
 * must be 16-byte aligned in a gated call.
 *   z       [tokens, Hv, dv] bf16, 16-byte aligned (tokens = B for decode)
 *   weight  [dv] f32, 16-byte aligned
 *   eps     >= 0 (1e-6 in Qwen3-Next)
 */
typedef enum { GDN_ACT_SILU = 0, GDN_ACT_SIGMOID = 1 } gdn_gate_act;
typedef struct {
  const void* z;
  const float* weight;
  float weight_offset;
  float eps;
  int32_t act; /* gdn_gate_act */
} gdn_output_gate;

/* Bits of the device error word (int32, caller-zeroed; the kernels only set
 * bits in it, with atomicOr, and never clear one). */
#define GDN_DEVERR_SLOT_RANGE 1 /* an active slot >= num_slots */
#define GDN_DEVERR_SEQLENS 2    /* cu_seqlens not non-decreasing or not ending at total_tokens */
#define GDN_DEVERR_TIMEOUT 4    /* a bounded wait (about a second) for an asynchronous copy or
                                   a tensor-core group gave up: the call's outputs and the
                                   states of its active slots are not to be trusted; slots the
                                   call does not address are untouched, and the context stays
                                   usable (include/gdn_testing.h makes one wait run out) */

/*
 * gdn_conv_update -- one decode step of the causal depthwise conv1d ([P1]
 * Summary, "The conv half of the decode step"; Notes, "The conv half").
 *
 * Per active row b (slot s = slot[b]) and channel c:
 *   win[0..W-2] = conv_state[s, c, :] (oldest first), win[W-1] = x[b, c]
 *   acc = bias[c] (or 0), in fp32; for j = 0..W-1:
 *       acc += round_to_operand_dtype(weight[c, j] * win[j])
 *   (bf16 cache: each product rounded to bf16; f32 cache: to f32)
 *   y = silu ? acc / (1 + exp(-acc)) : acc ;  out[b, c] = bf16(y)
 *   conv_state[s, c, :] <- win[1..W-1]          (a bit copy)
 *
 *   x          [B, D] bf16
 *   conv_state pool, in place: [num_slots, D, W-1] or [num_slots, W-1, D]
 *              (conv_layout) of state_dtype
 *   weight     [D, W] bf16 (tap W-1 multiplies the newest input)
 *   bias       [D] bf16, or NULL for none
 *   slot       [B] int32
 *   out        [B, D] bf16; inactive rows are written as zeros
 *   err        device int32 error word, or NULL
 * Supported: W == 4, D % 8 == 0. B == 0 is a no-op.
 */
gdn_status gdn_conv_update(const void* x, void* conv_state, gdn_dtype state_dtype,
                           gdn_conv_layout conv_layout, const void* weight, const void* bias,
                           int32_t silu, const int32_t* slot, int32_t batch, int32_t dim,
                           int32_t width, int32_t num_slots, void* out, int32_t* err,
                           void* stream);

/*
 * gdn_decode_step -- one fused decode step of the GDN layer: conv roll + conv
 * + SiLU, split into q|k|v, QK L2 norm, gating and the gated delta rule
 * ([P1] Summary: gating, QK norm "x / sqrt(sum(x*x) + 1e-6)" with scale on q
 * after the norm, no repeat_interleave, state ABI [num_blocks, HV, V, K]).
 *
 * Per active row b and value head h (k-head kh = h / (Hv/Hk)):
 *   q = conv(q channels of kh), k = conv(k channels of kh), v = conv(v of h)
 *   (bf16 after the conv, exactly as gdn_conv_update computes them)
 *   if qk_l2norm: q <- q / sqrt(sum q^2 + 1e-6) * scale, k <- k / sqrt(sum k^2 + 1e-6)
 *   else:         q <- q * scale
 *   a = exp(g), b = beta (gate_mode)
 *   S = ssm_state[s, h] ([dv, dk], dk contiguous)
 *   S <- a S;  d = b (v - S k);  S <- S + d k^T;  out[b, h] = S q
 *
 *   mixed_qkv   [B, D] bf16 (pre-conv; already q|k|v when conv_weight is NULL)
 *   a, b        gate inputs for [B, Hv] (see gdn_gate_mode)
 *   A_log, dt_bias  [Hv] f32 (FUSED mode)
 *   conv_weight [D, W] bf16, or NULL to bypass the conv (conv_state unused)
 *   conv_bias   [D] bf16 or NULL
 *   conv_state  conv pool as in gdn_conv_update, in place
 *   ssm_state   [num_slots, Hv, dv, dk] f32 (bf16 when dims.state_bf16), in place
 *   slot        [B] int32
 *   scale       multiplier applied to q (dk^-0.5 in Qwen3-Next)
 *   gate        NULL: out = o. Otherwise out = the gated RMSNorm of o (see
 *               gdn_output_gate), computed in the same kernel from the fp32 o
 *   out         [B, Hv, dv] of out_dtype (bf16 or f32); inactive rows zeroed
 * Supported: dk == dv in {32, 64, 128}, W == 4, Hv % Hk == 0, D % 8 == 0.
 */
gdn_status gdn_decode_step(const void* mixed_qkv, const void* a, const void* b,
                           gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                           const void* conv_weight, const void* conv_bias, int32_t silu,
                           void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                           float* ssm_state, const int32_t* slot, int32_t batch,
                           int32_t num_slots, gdn_dims dims, float scale, int32_t qk_l2norm,
                           const gdn_output_gate* gate, void* out, gdn_dtype out_dtype,
                           int32_t* err, void* stream);

/*
 * gdn_chunked_prefill_workspace_size -- bytes of device workspace that
 * gdn_chunked_prefill needs for these sizes (a host-side computation; 0 for
 * unsupported sizes).
 */
size_t gdn_chunked_prefill_workspace_size(int32_t total_tokens, int32_t num_seqs, gdn_dims dims,
                                          int32_t chunk);

/*
 * gdn_chunked_prefill -- the same layer over packed variable-length sequences
 * ([P4] "Numerical root cause and fix": per-chunk KK^T block, its
 * lower-triangular inverse, state passing). Mathematically identical to
 * running gdn_decode_step token by token over each sequence; it computes the
 * chunked (UT/WY) form with the triangular inverse solved exactly in fp32.
 *
 * Sequence i holds tokens [cu_seqlens[i], cu_seqlens[i+1]) of the packed
 * arrays and uses slot[i]. If has_initial_state is NULL or has_initial_state[i]
 * == 0, the sequence starts from a zero recurrent state and a zero conv window;
 * otherwise from ssm_state[slot] and conv_state[slot]. After the sequence, its
 * final recurrent state and final conv window (the last W-1 inputs of
 * initial window ++ x) are written to the slot. Inactive sequences (slot <= 0)
 * produce zero outputs and touch no state.
 *
 *   mixed_qkv   [total_tokens, D] bf16
 *   a, b        [total_tokens, Hv] gate inputs (gdn_gate_mode)
 *   cu_seqlens  [num_seqs + 1] int32, device: 0 = c0 <= c1 <= ... = total_tokens
 *   slot        [num_seqs] int32;  has_initial_state [num_seqs] uint8 or NULL
 *   out         [total_tokens, Hv, dv] of out_dtype; 16-byte aligned when gated, or when bf16
 *               with dk = dv = 128
 *   gate        NULL, or the output gate applied to every token's o (as in
 *               gdn_decode_step)
 *   chunk       chunk size C in {16, 32, 64}
 *   workspace   device scratch of >= gdn_chunked_prefill_workspace_size bytes,
 *               16-byte aligned; its contents on entry do not matter
 * Other arguments as in gdn_decode_step.
 * Supported: dk == dv in {32, 64, 128}, W == 4, Hv % Hk == 0, D % 8 == 0.
 *
 * With dk = dv = 128 and at most 64 (sequence, value head) pairs, the call runs its chunks in
 * pieces: several kernel launches on `stream`, the later ones programmatic dependents of the
 * ones before, so that each piece's state pass runs beside the next piece's intra-chunk
 * kernel. For the caller nothing changes: all of the call's work is ordered on `stream` as
 * before, and the results are bitwise those of one piece (the state crosses piece boundaries
 * in fp32, in the workspace).
 */
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
                               void* stream);

/*
 * gdn_chunked_prefill_noalloc -- gdn_chunked_prefill for callers that cannot
 * allocate device memory. The pages have no counterpart: this is a library
 * convenience, not part of the method.
 *
 * Who needs it: code that may not call an allocator (cudaMalloc can
 * synchronise the device, which a latency-critical host thread must not do), a
 * plug-in inside a runtime that owns every device allocation, or a process
 * that must keep a fixed device-memory footprint after start-up.
 *
 * It takes the same arguments as gdn_chunked_prefill minus the workspace: the
 * workspace lives in a fixed array of GDN_NOALLOC_SCRATCH_BYTES bytes in the
 * library's own device memory. The caller still owns and passes every input and
 * output. Limits:
 *   - every GPU on which the library is loaded holds that array until the
 *     process exits;
 *   - a call whose workspace (gdn_chunked_prefill_workspace_size) exceeds
 *     GDN_NOALLOC_SCRATCH_BYTES returns GDN_ERR_SCRATCH_LIMIT and enqueues
 *     nothing (64 MiB covers about 990 tokens of the Qwen3-Next geometry
 *     at chunk 64);
 *   - all calls on a device share the array: calls that may run at the same
 *     time on the GPU (streams without ordering between them) race on it;
 *   - the first call under each CUDA context looks up the array's device
 *     address (cudaGetSymbolAddress), which may load the module: make that
 *     first call before any stream capture. The address is kept per context;
 *     cudaDeviceReset is not supported after the first call (the primary
 *     context comes back under the same handle, with the array elsewhere).
 * Arguments are checked exactly as gdn_chunked_prefill checks them, and before
 * the look-up, so a bad call returns its status without any CUDA call.
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)

gdn_status gdn_chunked_prefill_noalloc(const void* mixed_qkv, const void* a, const void* b,
                                       gdn_gate_mode gate_mode, const float* A_log,
                                       const float* dt_bias, const void* conv_weight,
                                       const void* conv_bias, int32_t silu, void* conv_state,
                                       gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                                       float* ssm_state, const int32_t* cu_seqlens,
                                       const int32_t* slot, const uint8_t* has_initial_state,
                                       int32_t num_seqs, int32_t total_tokens, int32_t num_slots,
                                       gdn_dims dims, float scale, int32_t qk_l2norm,
                                       int32_t chunk, const gdn_output_gate* gate, void* out,
                                       gdn_dtype out_dtype, int32_t* err, void* stream);

/*
 * gdn_mixed_step -- one step that holds decode rows and prefill sequences
 * together, packed decode rows first (RL-Kernel PR #469 page, "Not
 * reproducible from this branch: the mixed decode+prefill measurement": a
 * provider that sends mixed-step decodes through another kernel makes their
 * results depend on the step's composition). Here the decode rows run the
 * fused decode kernel and the prefill sequences the chunked path, exactly as
 * gdn_decode_step and gdn_chunked_prefill would: every output, recurrent state
 * and conv state is bitwise the separate calls', whatever the mix.
 *
 * Packing: token rows [0, num_decode) are decode rows (one token each), rows
 * [num_decode, num_decode + prefill_tokens) the prefill sequences, for
 * mixed_qkv, a, b, out and the gate's z alike. slot holds num_decode +
 * num_prefill_seqs entries, decode rows first; cu_seqlens [num_prefill_seqs+1]
 * counts tokens from the start of the prefill part (0 ... prefill_tokens);
 * has_initial_state covers the prefill sequences. All active slots of the step
 * must be distinct. workspace is the prefill part's
 * (gdn_chunked_prefill_workspace_size(prefill_tokens, num_prefill_seqs, ...)).
 * Either part may be empty. Argument checks and result codes are those of the
 * two separate calls.
 *
 * Scheduling: the decode rows run on a library-owned side stream that waits
 * for the prefill's state pass to start (its last piece, when a prefill of few
 * sequences runs in pieces), on the SMs the pass leaves free; the
 * caller's stream then waits for the side stream, so the call is ordered on
 * `stream` like any other. The side stream and its events are created on the
 * first call per device that holds both parts: make it before any stream
 * capture. Mixed calls on one device enqueue one at a time.
 */
gdn_status gdn_mixed_step(const void* mixed_qkv, const void* a, const void* b,
                          gdn_gate_mode gate_mode, const float* A_log, const float* dt_bias,
                          const void* conv_weight, const void* conv_bias, int32_t silu,
                          void* conv_state, gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                          float* ssm_state, const int32_t* slot, int32_t num_decode,
                          const int32_t* cu_seqlens, const uint8_t* has_initial_state,
                          int32_t num_prefill_seqs, int32_t prefill_tokens, int32_t num_slots,
                          gdn_dims dims, float scale, int32_t qk_l2norm, int32_t chunk,
                          const gdn_output_gate* gate, void* out, gdn_dtype out_dtype,
                          void* workspace, size_t workspace_bytes, int32_t* err, void* stream);

/*
 * CUDA-graph decode buckets ([P2] Rocket, "A reduction barrier makes Qwen GDN
 * graph replay bit exact": immutable graphs per decode bucket c1, c2, ...,
 * inactive rows cleared on bucket transitions, slot 0 untouched).
 *
 * gdn_decode_graph_create captures ONE gdn_decode_step call -- same arguments
 * (the gate struct, if any, is read at creation; its z and weight buffers are
 * kept by pointer like every other buffer), same validation and the same
 * result codes -- into an instantiated CUDA graph
 * and returns it in *graph_out. Nothing runs at creation. The graph keeps the
 * pointers it was created with: the caller keeps those buffers alive and
 * unmoved, and writes each step's inputs (x, gate inputs, slot table) into
 * them before gdn_graph_launch. Rows a step does not use get slot 0, which makes
 * their outputs zero and leaves every state block alone. Creation is a set-up
 * call (it creates a stream and instantiates a graph); launching is not.
 * gdn_graph_launch enqueues the graph on `stream` (a cudaStream_t); a replay is
 * bitwise identical to the direct call. gdn_graph_destroy frees the handle
 * (NULL is ignored).
 */
typedef struct gdn_graph gdn_graph;

gdn_status gdn_decode_graph_create(const void* mixed_qkv, const void* a, const void* b,
                                   gdn_gate_mode gate_mode, const float* A_log,
                                   const float* dt_bias, const void* conv_weight,
                                   const void* conv_bias, int32_t silu, void* conv_state,
                                   gdn_dtype conv_dtype, gdn_conv_layout conv_layout,
                                   float* ssm_state, const int32_t* slot, int32_t batch,
                                   int32_t num_slots, gdn_dims dims, float scale,
                                   int32_t qk_l2norm, const gdn_output_gate* gate, void* out,
                                   gdn_dtype out_dtype, int32_t* err, gdn_graph** graph_out);
gdn_status gdn_graph_launch(gdn_graph* graph, void* stream);
void gdn_graph_destroy(gdn_graph* graph);

/*
 * gdn_validate_slots -- host-side check of a HOST slot table ([P1] Notes,
 * "State ABI": the goldens raise on an active index that is out of range or
 * repeated). Returns 0 if every active slot (> 0) is < num_slots and no
 * active slot repeats; 1 if one is out of range; 2 if one repeats.
 */
int32_t gdn_validate_slots(const int32_t* host_slot, int32_t n, int32_t num_slots);

/* Static description of a status code. */
const char* gdn_status_string(gdn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
