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

// y[t, :] = conv output of token t (bf16) for every token of an active sequence (the
// tokens of inactive ones are never read). A CTA covers a run of min(kConvRun, C) tokens
// inside one chunk (so within one sequence, found in the chunk table) and 2 kConvRunThreads
// channels; a thread keeps one channel pair for the run, so a warp reads 128 contiguous
// bytes of each input row: the conv parameters are loaded once, the window is built once
// (from x or, before the sequence start, the initial conv state) and then rolled in
// registers, and the input rows come kConvBatch at a time with the next batch in flight
// (the loads, 4 bytes each, need that depth to keep the memory system busy). The
// per-channel taps are conv_tap_sum's, as in the decode conv; the SiLU is silu_fast (the
// kernel is bound by instruction issue, and its bf16 output feeds the prefill, whose bound is
// far looser than the unit of bf16 it can move; the decode conv keeps the IEEE silu_f).
constexpr int kConvRun = 32;
constexpr int kConvBatch = 8;
constexpr int kConvRunThreads = 256;

// The W-1 taps before token t0 of channels c0, c0 + 1 (t0 in sequence i starting at bos):
// positions before bos come from the initial conv state, or are zero without one.
template <bool kF32Cache>
__device__ __forceinline__ void window2(const LayerArgs& a, const PrefillExtra& p, int i, int bos,
                                        int t0, int c0, float (&win)[2][kConvW - 1]) {
  const uint16_t* x = static_cast<const uint16_t*>(a.mixed);
  const bool init = (p.has_init == nullptr) || (p.has_init[i] != 0);
  const int64_t s = a.slot[i];
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) {
    const int pos = t0 - (kConvW - 1) + j;
    if (pos >= bos) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(x + static_cast<int64_t>(pos) * a.D + c0);
      win[0][j] = __uint_as_float(v << 16);
      win[1][j] = __uint_as_float(v & 0xFFFF0000u);
    } else if (!init) {
      win[0][j] = win[1][j] = 0.0f;
    } else {
      const int jj = (kConvW - 1) + (pos - bos);  // tap of the initial window
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int64_t idx = a.conv_layout == GDN_CONV_DIM_FIRST
                                ? (s * a.D + c0 + ch) * (kConvW - 1) + jj
                                : (s * (kConvW - 1) + jj) * a.D + c0 + ch;
        win[ch][j] = kF32Cache ? static_cast<const float*>(a.conv_state)[idx]
                               : bf2f(static_cast<const uint16_t*>(a.conv_state)[idx]);
      }
    }
  }
}

template <bool kF32Cache>
__global__ void __launch_bounds__(kConvRunThreads)
    prefill_conv_kernel(LayerArgs a, PrefillExtra p, const int32_t* meta,
                        const int32_t* chunk_off, const int32_t* chunk_seq, uint16_t* y) {
  const int run = min(kConvRun, p.chunk), runs = p.chunk / run;
  const int c = blockIdx.x / runs;
  if (c >= meta[0]) return;
  const int i = chunk_seq[c];
  const int bos = p.cu_seqlens[i], eos = p.cu_seqlens[i + 1];
  const int t0 = bos + (c - chunk_off[i]) * p.chunk + (blockIdx.x % runs) * run;
  const int n = min(run, eos - t0);
  const int c0 = (blockIdx.y * kConvRunThreads + threadIdx.x) * 2;
  if (n <= 0 || c0 >= a.D) return;
  const uint16_t* x = static_cast<const uint16_t*>(a.mixed) + c0;
  float2 w[kConvW], bias;  // (channel c0, channel c0 + 1) pairs
  {
    const uint16_t* wp = static_cast<const uint16_t*>(a.conv_w) + static_cast<int64_t>(c0) * kConvW;
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wp));  // [2 channels][4 taps]
    float wf[8];
    unpack8(wv, wf);
#pragma unroll
    for (int j = 0; j < kConvW; ++j) w[j] = make_float2(wf[j], wf[kConvW + j]);
    const uint16_t* bp = static_cast<const uint16_t*>(a.conv_b);
    bias = bp ? make_float2(bf2f(bp[c0]), bf2f(bp[c0 + 1])) : make_float2(0.0f, 0.0f);
  }
  auto load_x = [&](int k) {  // input row t0 + k (zeros past the run)
    return k < n ? __ldg(reinterpret_cast<const unsigned int*>(x + static_cast<int64_t>(t0 + k) * a.D))
                 : 0u;
  };
  uint32_t xn[kConvBatch];
#pragma unroll
  for (int k = 0; k < kConvBatch; ++k) xn[k] = load_x(k);
  float2 win[kConvW];  // taps 0 .. W-2 of the current token, then its input
  {
    float w2[2][kConvW - 1];
    window2<kF32Cache>(a, p, i, bos, t0, c0, w2);
#pragma unroll
    for (int j = 0; j < kConvW - 1; ++j) win[j] = make_float2(w2[0][j], w2[1][j]);
  }
  uint16_t* yo = y + static_cast<int64_t>(t0) * a.D + c0;
  const bool silu = a.silu != 0;
#pragma unroll 1
  for (int kb = 0; kb < n; kb += kConvBatch) {
    uint32_t xc[kConvBatch];
#pragma unroll
    for (int k = 0; k < kConvBatch; ++k) {
      xc[k] = xn[k];
      xn[k] = load_x(kb + kConvBatch + k);
    }
#pragma unroll
    for (int k = 0; k < kConvBatch; ++k) {
      if (kb + k >= n) break;
      win[kConvW - 1] = make_float2(__uint_as_float(xc[k] << 16), __uint_as_float(xc[k] & 0xFFFF0000u));
      float2 acc = conv_tap_sum2<kF32Cache>(win, w, bias);
      if (silu) acc = make_float2(silu_fast(acc.x), silu_fast(acc.y));
#pragma unroll
      for (int j = 0; j < kConvW - 1; ++j) win[j] = win[j + 1];
      *reinterpret_cast<uint32_t*>(yo + static_cast<int64_t>(kb + k) * a.D) = pack_bf2(acc.x, acc.y);
    }
  }
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

cudaError_t launch_prefill_conv(const LayerArgs& a, const PrefillExtra& p, const int32_t* meta,
                                const int32_t* seq_ok, const int32_t* chunk_off,
                                const int32_t* chunk_seq, int max_chunks, uint16_t* y,
                                cudaStream_t s) {
  const int groups = a.D / 8;
  const int gy = (groups + kConvThreads - 1) / kConvThreads;
  if (max_chunks > 0) {
    dim3 grid(static_cast<unsigned>(max_chunks) * (p.chunk / min(kConvRun, p.chunk)),
              (a.D / 2 + kConvRunThreads - 1) / kConvRunThreads);
    if (a.conv_f32)
      prefill_conv_kernel<true><<<grid, kConvRunThreads, 0, s>>>(a, p, meta, chunk_off, chunk_seq, y);
    else
      prefill_conv_kernel<false><<<grid, kConvRunThreads, 0, s>>>(a, p, meta, chunk_off, chunk_seq, y);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 grid2(p.num_seqs, gy);
  if (a.conv_f32) prefill_conv_state_kernel<true><<<grid2, kConvThreads, 0, s>>>(a, p, seq_ok);
  else prefill_conv_state_kernel<false><<<grid2, kConvThreads, 0, s>>>(a, p, seq_ok);
  return cudaGetLastError();
}

}  // namespace gdn
