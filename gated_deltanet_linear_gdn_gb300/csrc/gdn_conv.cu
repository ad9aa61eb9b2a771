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

// y[t, :] = conv output of token t (bf16) for every token of an active sequence (the
// tokens of inactive ones are never read). A CTA covers a run of min(kConvRun, C) tokens
// inside one chunk (so within one sequence, found in the chunk table) and 8 kConvRunThreads
// channels; a thread keeps 8 consecutive channels for the run, so each of its input and
// output rows is one 16-byte access and a warp moves 512 contiguous bytes of a row. The conv
// parameters are loaded once, the window is built once (from x or, before the sequence start,
// the initial conv state) and then rolled in registers, and the input rows come kBatch at a
// time with the next batch in flight.
// Per channel the taps are conv_tap_sum's (fp32 accumulator from the bias, taps in order).
// With a bf16 cache every operand is a bf16 value, so each tap product rounded to bf16 is one
// packed bf16 multiply of the raw input words (the exact product, rounded once to nearest
// even, as the fp32 product -- exact for two bf16 factors -- rounded to bf16 is), added to the
// fp32 accumulator by a mixed-precision add that takes the bf16 half directly; with an fp32
// cache the products are fp32 (the initial window's values need not be bf16). The SiLU is
// silu_fast (the kernel is bound by instruction issue and memory, and its bf16 output feeds
// the prefill, whose bound is far looser than the unit of bf16 it can move; the decode conv
// keeps the IEEE silu_f).
constexpr int kConvRun = 32;
constexpr int kConvRunThreads = 256;
constexpr int kConvBatch = 8;

// two bf16 values (lo, hi) times two bf16 values, each product rounded to bf16
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}
// acc + (lo, hi) of a bf16 pair, each sum rounded once in fp32 (the bf16 operand converts
// exactly), as an fp32 add of the unpacked pair rounds it
__device__ __forceinline__ float2 add_bf16x2(float2 acc, uint32_t v) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y) : "r"(v));
  return acc;
}

// The W-1 taps before token t0 of channels [c0, c0 + 8) (t0 in sequence i starting at bos, a
// run start: bos itself or at least 16 tokens later): at the sequence start they are the
// initial conv state (zero without one), otherwise the W-1 input rows before t0.
template <bool kF32Cache>
__device__ __forceinline__ void window_before8(const LayerArgs& a, const PrefillExtra& p, int i,
                                               int bos, int t0, int c0,
                                               float (&win)[8][kConvW - 1]) {
  if (t0 == bos) {
    const bool init = (p.has_init == nullptr) || (p.has_init[i] != 0);
    if (init) {
      load_conv8<kF32Cache>(a.conv_state, a.conv_layout, a.slot[i], a.D, c0, win);
    } else {
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
#pragma unroll
        for (int j = 0; j < kConvW - 1; ++j) win[ch][j] = 0.0f;
    }
    return;
  }
  const uint16_t* x = static_cast<const uint16_t*>(a.mixed);
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) {
    float v[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t0 - (kConvW - 1) + j) * a.D + c0)), v);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) win[ch][j] = v[ch];
  }
}

template <bool kF32Cache, int kBatch>
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
  const int c0 = (blockIdx.y * kConvRunThreads + threadIdx.x) * 8;
  if (n <= 0 || c0 >= a.D) return;
  const uint16_t* x = static_cast<const uint16_t*>(a.mixed) + c0;
  // parameters: tap j of the channel pair (c0 + 2q, c0 + 2q + 1)
  uint32_t wq[kConvW][4];  // as bf16 pairs (lo = channel c0 + 2q)
  float2 bias[4];
  {
    const uint4* wp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.conv_w) +
                                                     static_cast<int64_t>(c0) * kConvW);
    uint32_t wa[16];  // [8 channels][4 taps] bf16, two per word
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(wp + k);
      wa[4 * k] = v.x; wa[4 * k + 1] = v.y; wa[4 * k + 2] = v.z; wa[4 * k + 3] = v.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int j = 0; j < kConvW; ++j)
        wq[j][q] = __byte_perm(wa[4 * q + (j >> 1)], wa[4 * q + 2 + (j >> 1)],
                               (j & 1) ? 0x7632 : 0x5410);
    const uint16_t* bp = static_cast<const uint16_t*>(a.conv_b);
    if (bp) {
      const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bp + c0));
      bias[0] = bf16x2_to_float2(bv.x); bias[1] = bf16x2_to_float2(bv.y);
      bias[2] = bf16x2_to_float2(bv.z); bias[3] = bf16x2_to_float2(bv.w);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) bias[q] = make_float2(0.0f, 0.0f);
    }
  }
  auto load_x = [&](int k) {  // input row t0 + k (zeros past the run)
    return k < n ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t0 + k) * a.D))
                 : make_uint4(0u, 0u, 0u, 0u);
  };
  uint4 xn[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k) xn[k] = load_x(k);
  // taps 0 .. W-2 of the current token: bf16 pairs (bf16 cache) or floats (fp32 cache)
  uint32_t wb[kConvW - 1][4];
  float2 wf[kConvW - 1][4];
  {
    float w8[8][kConvW - 1];
    window_before8<kF32Cache>(a, p, i, bos, t0, c0, w8);
#pragma unroll
    for (int j = 0; j < kConvW - 1; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wf[j][q] = make_float2(w8[2 * q][j], w8[2 * q + 1][j]);
        wb[j][q] = pack_bf2(w8[2 * q][j], w8[2 * q + 1][j]);  // exact: bf16 values
      }
  }
  uint16_t* yo = y + static_cast<int64_t>(t0) * a.D + c0;
  const bool silu = a.silu != 0;
#pragma unroll 1
  for (int kb = 0; kb < n; kb += kBatch) {
    uint4 xc[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      xc[k] = xn[k];
      xn[k] = load_x(kb + kBatch + k);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (kb + k >= n) break;
      const uint32_t xw[4] = {xc[k].x, xc[k].y, xc[k].z, xc[k].w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float2 acc = bias[q];
        if (!kF32Cache) {
#pragma unroll
          for (int j = 0; j < kConvW; ++j)
            acc = add_bf16x2(acc, mul_bf16x2(wq[j][q], j < kConvW - 1 ? wb[j][q] : xw[q]));
        } else {
          const float2 xf = bf16x2_to_float2(xw[q]);
#pragma unroll
          for (int j = 0; j < kConvW; ++j)
            acc = __fadd2_rn(acc, __fmul2_rn(bf16x2_to_float2(wq[j][q]), j < kConvW - 1 ? wf[j][q] : xf));
        }
        if (silu) acc = make_float2(silu_fast(acc.x), silu_fast(acc.y));
        o[q] = pack_bf2(acc.x, acc.y);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!kF32Cache) {
#pragma unroll
          for (int j = 0; j < kConvW - 2; ++j) wb[j][q] = wb[j + 1][q];
          wb[kConvW - 2][q] = xw[q];
        } else {
#pragma unroll
          for (int j = 0; j < kConvW - 2; ++j) wf[j][q] = wf[j + 1][q];
          wf[kConvW - 2][q] = bf16x2_to_float2(xw[q]);
        }
      }
      *reinterpret_cast<uint4*>(yo + static_cast<int64_t>(kb + k) * a.D) = make_uint4(o[0], o[1], o[2], o[3]);
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
              (a.D / 8 + kConvRunThreads - 1) / kConvRunThreads);
    if (a.conv_f32)
      prefill_conv_kernel<true, kConvBatch><<<grid, kConvRunThreads, 0, s>>>(a, p, meta, chunk_off,
                                                                             chunk_seq, y);
    else
      prefill_conv_kernel<false, kConvBatch><<<grid, kConvRunThreads, 0, s>>>(a, p, meta, chunk_off,
                                                                              chunk_seq, y);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 grid2(p.num_seqs, gy);
  if (a.conv_f32) prefill_conv_state_kernel<true><<<grid2, kConvThreads, 0, s>>>(a, p, seq_ok);
  else prefill_conv_state_kernel<false><<<grid2, kConvThreads, 0, s>>>(a, p, seq_ok);
  return cudaGetLastError();
}

}  // namespace gdn
