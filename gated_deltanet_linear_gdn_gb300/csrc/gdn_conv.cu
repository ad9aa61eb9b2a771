// gdn_conv.cu -- causal depthwise conv1d kernels (width 4) for decode and
// prefill. RL-Kernel PR #469 "C6: GDN decode-step goldens and recurrent/conv
// state contract": Summary (conv bullet: fp32 accumulator from the bias, tap
// products rounded to the operand dtype) and Notes "State ABI" (slots <= 0
// skipped with zero output, conv state [num_blocks, dim, W-1] or transposed).
//
// Each thread owns 8 consecutive channels of one row/token: 16-byte loads of
// x, weight and bias, and 16-byte-aligned conv-state loads/stores (48 or 96
// contiguous bytes in the dim-first layout). The kernels are HBM-bound.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kConvThreads = 128;

template <bool kF32Cache>
__global__ void __launch_bounds__(kConvThreads) conv_update_kernel(ConvUpdateArgs a) {
  const int b = blockIdx.y;
  const int g = blockIdx.x * kConvThreads + threadIdx.x;
  const int c0 = g * 8;
  if (c0 >= a.D) return;
  const int32_t s = a.slot[b];
  uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + static_cast<int64_t>(b) * a.D + c0);
  if (s <= 0 || s >= a.num_slots) {
    if (s >= a.num_slots && g == 0 && a.err) atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
    *out = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  float win[8][kConvW - 1];
  load_conv8<kF32Cache>(a.conv_state, a.layout, s, a.D, c0, win);
  float x8[8];
  unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) +
                                                static_cast<int64_t>(b) * a.D + c0)), x8);
  float y8[8];
  conv8_step<kF32Cache>(win, x8, static_cast<const uint16_t*>(a.weight),
                        static_cast<const uint16_t*>(a.bias), c0, a.silu != 0, y8);
  store_conv8<kF32Cache>(a.conv_state, a.layout, s, a.D, c0, win);
  uint16_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = f2bf(y8[i]);
  *out = pack8(h);
}

__device__ __forceinline__ int find_seq(const int32_t* cu, int n, int t) {
  // largest i with cu[i] <= t (cu non-decreasing; cu[0] = 0 <= t < cu[n])
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Window tap j of token t: position p = t - (W-1) + j of its sequence; before
// the sequence start it comes from the initial conv state (or zero).
template <bool kF32Cache>
__device__ __forceinline__ void window8(const LayerArgs& a, const PrefillExtra& p, int i, int bos,
                                        int t, int c0, float (&win)[8][kConvW - 1],
                                        float (&x8)[8]) {
  const uint16_t* x = static_cast<const uint16_t*>(a.mixed);
  const bool init = (p.has_init == nullptr) || (p.has_init[i] != 0);
  const int32_t s = a.slot[i];
  bool need_init = false;
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) need_init |= (t - (kConvW - 1) + j < bos);
  float st[8][kConvW - 1];
  if (need_init && init) load_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, st);
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) {
    const int pos = t - (kConvW - 1) + j;
    if (pos >= bos) {
      float v[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(pos) * a.D + c0)), v);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) win[ch][j] = v[ch];
    } else {
      const int jj = (kConvW - 1) + (pos - bos);  // 0..W-2
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) win[ch][j] = init ? st[ch][jj] : 0.0f;
    }
  }
  unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * a.D + c0)), x8);
}

// y[t, :] = conv output of token t (bf16). One block per token.
template <bool kF32Cache>
__global__ void __launch_bounds__(kConvThreads)
    prefill_conv_kernel(LayerArgs a, PrefillExtra p, const int32_t* seq_ok, uint16_t* y) {
  __shared__ int s_seq;
  const int t = blockIdx.x;
  if (threadIdx.x == 0) s_seq = find_seq(p.cu_seqlens, p.num_seqs, t);
  __syncthreads();
  const int i = s_seq;
  const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * 8;
  if (c0 >= a.D) return;
  uint4* yo = reinterpret_cast<uint4*>(y + static_cast<int64_t>(t) * a.D + c0);
  if (!seq_ok[i]) {
    *yo = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int bos = p.cu_seqlens[i];
  float win[8][kConvW - 1], x8[8], y8[8];
  window8<kF32Cache>(a, p, i, bos, t, c0, win, x8);
  conv8_step<kF32Cache>(win, x8, static_cast<const uint16_t*>(a.conv_w),
                        static_cast<const uint16_t*>(a.conv_b), c0, a.silu != 0, y8);
  uint16_t h[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = f2bf(y8[k]);
  *yo = pack8(h);
}

// Final conv window of each sequence = last W-1 entries of (initial ++ x).
// Runs after prefill_conv_kernel (same stream), which read the initial state.
template <bool kF32Cache>
__global__ void __launch_bounds__(kConvThreads)
    prefill_conv_state_kernel(LayerArgs a, PrefillExtra p, const int32_t* seq_ok) {
  const int i = blockIdx.x;
  const int c0 = (blockIdx.y * kConvThreads + threadIdx.x) * 8;
  if (c0 >= a.D || !seq_ok[i]) return;
  const int bos = p.cu_seqlens[i], eos = p.cu_seqlens[i + 1];
  float win[8][kConvW - 1], x8[8];
  // the window a token at position eos would see: taps j = 0..W-2 at eos-(W-1)+j
  const uint16_t* x = static_cast<const uint16_t*>(a.mixed);
  const bool init = (p.has_init == nullptr) || (p.has_init[i] != 0);
  float st[8][kConvW - 1];
  if (init && eos - (kConvW - 1) < bos)
    load_conv8<kF32Cache>(a.conv_state, a.conv_layout, a.slot[i], a.D, c0, st);
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) {
    const int pos = eos - (kConvW - 1) + j;
    if (pos >= bos) {
      float v[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(pos) * a.D + c0)), v);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) win[ch][j] = v[ch];
    } else {
      const int jj = (kConvW - 1) + (pos - bos);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) win[ch][j] = init ? st[ch][jj] : 0.0f;
    }
  }
  (void)x8;
  store_conv8<kF32Cache>(a.conv_state, a.conv_layout, a.slot[i], a.D, c0, win);
}

}  // namespace

cudaError_t launch_conv_update(const ConvUpdateArgs& a, cudaStream_t s) {
  const int groups = a.D / 8;
  dim3 grid((groups + kConvThreads - 1) / kConvThreads, a.B);
  if (a.f32_cache) conv_update_kernel<true><<<grid, kConvThreads, 0, s>>>(a);
  else conv_update_kernel<false><<<grid, kConvThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_conv(const LayerArgs& a, const PrefillExtra& p, const int32_t* seq_ok,
                                uint16_t* y, cudaStream_t s) {
  const int groups = a.D / 8;
  const int gy = (groups + kConvThreads - 1) / kConvThreads;
  if (p.total_tokens > 0) {
    dim3 grid(p.total_tokens, gy);
    if (a.conv_f32) prefill_conv_kernel<true><<<grid, kConvThreads, 0, s>>>(a, p, seq_ok, y);
    else prefill_conv_kernel<false><<<grid, kConvThreads, 0, s>>>(a, p, seq_ok, y);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 grid2(p.num_seqs, gy);
  if (a.conv_f32) prefill_conv_state_kernel<true><<<grid2, kConvThreads, 0, s>>>(a, p, seq_ok);
  else prefill_conv_state_kernel<false><<<grid2, kConvThreads, 0, s>>>(a, p, seq_ok);
  return cudaGetLastError();
}

}  // namespace gdn
