// gdn_common.cuh -- device helpers shared by the GDN kernels (sm_103a).
//
// Conv arithmetic follows RL-Kernel PR #469 "C6: GDN decode-step goldens and
// recurrent/conv state contract", Summary (conv bullet): an fp32 accumulator
// that starts from the bias, every tap product rounded to the operand dtype
// before it is added. Adds and multiplies use the explicit _rn intrinsics so
// that no FMA contraction changes the rounding.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kConvW = 4;  // conv width supported by the kernels

__device__ __forceinline__ float bf2f(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}
__device__ __forceinline__ float round_bf(float f) { return bf2f(f2bf(f)); }
// Two floats -> two bf16 (round to nearest even) in one word, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Unpack 8 bf16 values held in a uint4.
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack8(const uint16_t* h) {
  uint4 u;
  u.x = h[0] | (static_cast<uint32_t>(h[1]) << 16);
  u.y = h[2] | (static_cast<uint32_t>(h[3]) << 16);
  u.z = h[4] | (static_cast<uint32_t>(h[5]) << 16);
  u.w = h[6] | (static_cast<uint32_t>(h[7]) << 16);
  return u;
}

// One conv output: acc = bias + sum_j round_op(w_j * win_j) in fp32, then
// optional SiLU (expf and IEEE division), returned before the bf16 store.
template <bool kF32Cache>
__device__ __forceinline__ float conv_tap_sum(const float (&win)[kConvW], const float (&w)[kConvW],
                                              float bias) {
  float acc = bias;
#pragma unroll
  for (int j = 0; j < kConvW; ++j) {
    float p = __fmul_rn(w[j], win[j]);
    if (!kF32Cache) p = round_bf(p);
    acc = __fadd_rn(acc, p);
  }
  return acc;
}

// conv_tap_sum for two channels at once, in packed f32x2 operations: per channel the same
// roundings in the same order (so the same results), half the instructions for the taps.
template <bool kF32Cache>
__device__ __forceinline__ float2 conv_tap_sum2(const float2 (&win)[kConvW], const float2 (&w)[kConvW],
                                                float2 bias) {
  float2 acc = bias;
#pragma unroll
  for (int j = 0; j < kConvW; ++j) {
    float2 p = __fmul2_rn(w[j], win[j]);
    if (!kF32Cache) {
      const uint32_t h = pack_bf2(p.x, p.y);
      p = make_float2(__uint_as_float(h << 16), __uint_as_float(h & 0xFFFF0000u));
    }
    acc = __fadd2_rn(acc, p);
  }
  return acc;
}

__device__ __forceinline__ float silu_f(float x) { return __fdiv_rn(x, __fadd_rn(1.0f, expf(-x))); }
// The same with the hardware exponential and a fast division (a few ulp of fp32 from silu_f;
// the bf16 value it rounds to differs from silu_f's in about one element in 10^4, by one unit).
// x below about -88 gives 1 + e^-x = inf and the quotient 0, as the exact SiLU tends to.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// ---------------------------------------------------------------------------
// Conv state access for 8 consecutive channels [c0, c0+8) of one slot.
// DIM_FIRST: [slots, D, 3] -> 24 contiguous entries; TAP_FIRST: [slots, 3, D].
// win[ch][j], j = 0 oldest. Requires c0 % 8 == 0 and a 16-byte aligned pool.
// ---------------------------------------------------------------------------
// The packed window of 8 channels (24 values in the pool dtype) as 16-byte words,
// so that several groups' loads can be in flight before any is unpacked.
template <bool kF32Cache>
struct RawWin8 {
  uint4 v[kF32Cache ? 6 : 3];
};

template <bool kF32Cache>
__device__ __forceinline__ void load_conv8_raw(const void* pool, int layout, int64_t slot, int D,
                                               int c0, RawWin8<kF32Cache>& r) {
  constexpr int kEs = kF32Cache ? 4 : 2;
  const char* base = static_cast<const char*>(pool);
  if (layout == GDN_CONV_DIM_FIRST) {
    const uint4* p = reinterpret_cast<const uint4*>(base + (slot * D + c0) * (kConvW - 1) * kEs);
#pragma unroll
    for (int i = 0; i < (kF32Cache ? 6 : 3); ++i) r.v[i] = p[i];
  } else {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const uint4* p = reinterpret_cast<const uint4*>(base + ((slot * (kConvW - 1) + j) * D + c0) * kEs);
      if (kF32Cache) {
        r.v[2 * j] = p[0];
        r.v[2 * j + 1] = p[1];
      } else {
        r.v[j] = p[0];
      }
    }
  }
}

template <bool kF32Cache>
__device__ __forceinline__ void unpack_conv8(const RawWin8<kF32Cache>& r, int layout,
                                             float (&win)[8][kConvW - 1]) {
  if (layout == GDN_CONV_DIM_FIRST) {  // 24 values in (channel, tap) order
    float v[24];
#pragma unroll
    for (int i = 0; i < (kF32Cache ? 6 : 3); ++i) {
      if (kF32Cache) {
        v[4 * i] = __uint_as_float(r.v[i].x); v[4 * i + 1] = __uint_as_float(r.v[i].y);
        v[4 * i + 2] = __uint_as_float(r.v[i].z); v[4 * i + 3] = __uint_as_float(r.v[i].w);
      } else {
        unpack8(r.v[i], v + 8 * i);
      }
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
#pragma unroll
      for (int j = 0; j < 3; ++j) win[ch][j] = v[3 * ch + j];
  } else {  // one 8-channel vector per tap
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      float v[8];
      if (kF32Cache) {
        const uint4 a = r.v[2 * j], b = r.v[2 * j + 1];
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
        v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
        v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
      } else {
        unpack8(r.v[j], v);
      }
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) win[ch][j] = v[ch];
    }
  }
}

template <bool kF32Cache>
__device__ __forceinline__ void load_conv8(const void* pool, int layout, int64_t slot, int D, int c0,
                                           float (&win)[8][kConvW - 1]) {
  RawWin8<kF32Cache> r;
  load_conv8_raw<kF32Cache>(pool, layout, slot, D, c0, r);
  unpack_conv8<kF32Cache>(r, layout, win);
}

// Store a window whose values are exactly representable in the pool dtype.
template <bool kF32Cache>
__device__ __forceinline__ void store_conv8(void* pool, int layout, int64_t slot, int D, int c0,
                                            const float (&win)[8][kConvW - 1]) {
  if (layout == GDN_CONV_DIM_FIRST) {
    if (kF32Cache) {
      float4* p = reinterpret_cast<float4*>(static_cast<float*>(pool) + (slot * D + c0) * (kConvW - 1));
      float v[24];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
#pragma unroll
        for (int j = 0; j < 3; ++j) v[3 * ch + j] = win[ch][j];
#pragma unroll
      for (int i = 0; i < 6; ++i) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
      uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(pool) + (slot * D + c0) * (kConvW - 1));
      uint16_t h[24];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
#pragma unroll
        for (int j = 0; j < 3; ++j) h[3 * ch + j] = f2bf(win[ch][j]);
#pragma unroll
      for (int i = 0; i < 3; ++i) p[i] = pack8(h + 8 * i);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int64_t off = (slot * (kConvW - 1) + j) * D + c0;
      if (kF32Cache) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(pool) + off);
        p[0] = make_float4(win[0][j], win[1][j], win[2][j], win[3][j]);
        p[1] = make_float4(win[4][j], win[5][j], win[6][j], win[7][j]);
      } else {
        uint16_t h[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) h[ch] = f2bf(win[ch][j]);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(pool) + off) = pack8(h);
      }
    }
  }
}

// Conv weights [8 channels][4 taps] and bias of one 8-channel group, packed bf16.
struct ConvParams8 {
  uint4 w[4];
  uint4 b;
};
__device__ __forceinline__ ConvParams8 conv8_params(const uint16_t* __restrict__ weight,
                                                    const uint16_t* __restrict__ bias, int c0) {
  ConvParams8 p;
  const uint4* wp = reinterpret_cast<const uint4*>(weight + static_cast<int64_t>(c0) * kConvW);
#pragma unroll
  for (int i = 0; i < 4; ++i) p.w[i] = __ldg(wp + i);
  p.b = bias ? __ldg(reinterpret_cast<const uint4*>(bias + c0)) : make_uint4(0u, 0u, 0u, 0u);
  return p;
}

// Conv of 8 channels for one new input vector x8 with loaded parameters; rolls
// win in place and returns the bf16-rounded outputs as floats. (A missing bias
// loads as +0, the accumulator's start value either way.)
template <bool kF32Cache>
__device__ __forceinline__ void conv8_apply(float (&win)[8][kConvW - 1], const float (&x8)[8],
                                            const ConvParams8& prm, bool silu, float (&y8)[8]) {
  float w[32], bv[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack8(prm.w[i], w + 8 * i);
  unpack8(prm.b, bv);
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    float full[kConvW] = {win[ch][0], win[ch][1], win[ch][2], x8[ch]};
    float wc[kConvW] = {w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]};
    float acc = conv_tap_sum<kF32Cache>(full, wc, bv[ch]);
    if (silu) acc = silu_f(acc);
    y8[ch] = round_bf(acc);
    win[ch][0] = full[1];
    win[ch][1] = full[2];
    win[ch][2] = full[3];
  }
}

// Conv of 8 channels [c0, c0+8) for one new input vector x8; rolls win in
// place and returns the bf16-rounded outputs as floats.
template <bool kF32Cache>
__device__ __forceinline__ void conv8_step(float (&win)[8][kConvW - 1], const float (&x8)[8],
                                           const uint16_t* __restrict__ weight,
                                           const uint16_t* __restrict__ bias, int c0, bool silu,
                                           float (&y8)[8]) {
  conv8_apply<kF32Cache>(win, x8, conv8_params(weight, bias, c0), silu, y8);
}

// ---------------------------------------------------------------------------
// Gating (RL-Kernel PR #469, Notes "How the golden relates to the kernel",
// item 1): fp32, softplus threshold at 20.
// ---------------------------------------------------------------------------
// The raw gate inputs of one (token, head), loaded ahead of their arithmetic so the
// loads can overlap other work; gate_from_raw turns them into alpha = exp(g), beta.
struct GateRaw {
  float a, b, A_log, dt_bias;
};
__device__ __forceinline__ GateRaw gate_load(const void* a, const void* b, int gate_mode,
                                             const float* A_log, const float* dt_bias,
                                             int64_t idx, int h) {
  GateRaw r;
  if (gate_mode == GDN_GATE_DIRECT) {
    r.a = static_cast<const float*>(a)[idx];
    r.b = static_cast<const float*>(b)[idx];
    r.A_log = r.dt_bias = 0.0f;
  } else {
    r.a = bf2f(static_cast<const uint16_t*>(a)[idx]);
    r.b = bf2f(static_cast<const uint16_t*>(b)[idx]);
    r.A_log = A_log[h];
    r.dt_bias = dt_bias[h];
  }
  return r;
}
__device__ __forceinline__ void gate_from_raw(const GateRaw& r, int gate_mode, float& alpha,
                                              float& beta) {
  if (gate_mode == GDN_GATE_DIRECT) {
    beta = r.b;
    alpha = expf(r.a);
  } else {
    const float x = __fadd_rn(r.a, r.dt_bias);
    const float sp = x > 20.0f ? x : log1pf(expf(x));
    const float g = __fmul_rn(-expf(r.A_log), sp);
    alpha = expf(g);
    beta = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-r.b)));
  }
}

// log-space variant used by the chunked prefill (it needs g itself), from loaded inputs.
__device__ __forceinline__ void gate_log_raw(const GateRaw& r, int gate_mode, float& g,
                                             float& beta) {
  if (gate_mode == GDN_GATE_DIRECT) {
    g = r.a;
    beta = r.b;
  } else {
    const float x = __fadd_rn(r.a, r.dt_bias);
    const float sp = x > 20.0f ? x : log1pf(expf(x));
    g = __fmul_rn(-expf(r.A_log), sp);
    beta = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-r.b)));
  }
}

// log-space variant used by the chunked prefill (it needs g itself).
__device__ __forceinline__ void gate_log(const void* a, const void* b, int gate_mode,
                                         const float* A_log, const float* dt_bias, int64_t idx,
                                         int h, float& g, float& beta) {
  if (gate_mode == GDN_GATE_DIRECT) {
    g = static_cast<const float*>(a)[idx];
    beta = static_cast<const float*>(b)[idx];
  } else {
    const float x = __fadd_rn(bf2f(static_cast<const uint16_t*>(a)[idx]), dt_bias[h]);
    const float sp = x > 20.0f ? x : log1pf(expf(x));
    g = __fmul_rn(-expf(A_log[h]), sp);
    beta = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-bf2f(static_cast<const uint16_t*>(b)[idx]))));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace gdn
