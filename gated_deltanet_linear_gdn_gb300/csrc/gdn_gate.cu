// gdn_gate.cu -- the GDN block's output gate over stored rows: a gated RMSNorm
// of each (token, value head) vector of `out`, in place (RL-Kernel PR #469
// "C6: GDN decode-step goldens and recurrent/conv state contract", Summary by
// CodeRabbit and Walkthrough, on the stacked gated-RMSNorm PRs #466-#468: SiLU
// or sigmoid gating and a weight offset). The chunked prefill runs it after its state
// pass; the decode step fuses the same arithmetic into its own epilogue warp.
//
// Per row (dv values o, the matching z):
//   out = o / sqrt(mean(o^2) + eps) * (w + offset) * act(z)
// in fp32 from o as stored (a bf16 output is read back as bf16, which is the
// block's unfused arithmetic), an all-zero row with eps 0 giving zero. The
// activation takes the hardware exponential and a fast quotient (silu_fast; the
// sigmoid likewise): the kernel is bound by instruction issue, and the prefill's
// bound is far looser than the few fp32 ulp this moves. The decode epilogue keeps
// the IEEE forms.
//
// One warp per row, dv/32 consecutive elements per lane, a 5-step xor-shuffle
// sum of squares; a grid-stride loop over rows (kGateRows = 1: more rows in
// flight per warp cost occupancy and measured slower). Per row it reads o and z
// and writes y.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kGateWarps = 8;
constexpr int kGateRows = 1;  // consecutive rows a warp takes at a time

template <int VPL>
struct RowIO;
template <>
struct RowIO<4> {
  static __device__ void load_bf16(const uint16_t* p, int lane, float (&v)[4]) {
    const uint2 u = reinterpret_cast<const uint2*>(p)[lane];
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
  static __device__ void store_bf16(uint16_t* p, int lane, const float (&v)[4]) {
    reinterpret_cast<uint2*>(p)[lane] = make_uint2(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]));
  }
  static __device__ void load_f32(const float* p, int lane, float (&v)[4]) {
    const float4 f = reinterpret_cast<const float4*>(p)[lane];
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
  static __device__ void store_f32(float* p, int lane, const float (&v)[4]) {
    reinterpret_cast<float4*>(p)[lane] = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct RowIO<2> {
  static __device__ void load_bf16(const uint16_t* p, int lane, float (&v)[2]) {
    const uint32_t u = reinterpret_cast<const uint32_t*>(p)[lane];
    v[0] = __uint_as_float(u << 16); v[1] = __uint_as_float(u & 0xFFFF0000u);
  }
  static __device__ void store_bf16(uint16_t* p, int lane, const float (&v)[2]) {
    reinterpret_cast<uint32_t*>(p)[lane] = pack_bf2(v[0], v[1]);
  }
  static __device__ void load_f32(const float* p, int lane, float (&v)[2]) {
    const float2 f = reinterpret_cast<const float2*>(p)[lane];
    v[0] = f.x; v[1] = f.y;
  }
  static __device__ void store_f32(float* p, int lane, const float (&v)[2]) {
    reinterpret_cast<float2*>(p)[lane] = make_float2(v[0], v[1]);
  }
};
template <>
struct RowIO<1> {
  static __device__ void load_bf16(const uint16_t* p, int lane, float (&v)[1]) { v[0] = bf2f(p[lane]); }
  static __device__ void store_bf16(uint16_t* p, int lane, const float (&v)[1]) { p[lane] = f2bf(v[0]); }
  static __device__ void load_f32(const float* p, int lane, float (&v)[1]) { v[0] = p[lane]; }
  static __device__ void store_f32(float* p, int lane, const float (&v)[1]) { p[lane] = v[0]; }
};

template <int VPL>
__global__ void __launch_bounds__(32 * kGateWarps)
    gate_rows_kernel(LayerArgs a, int64_t rows) {
  constexpr int DV = 32 * VPL;
  using IO = RowIO<VPL>;
  const int lane = threadIdx.x & 31;
  float w[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) w[e] = __ldg(a.gate_w + lane * VPL + e) + a.gate_offset;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kGateWarps * kGateRows;
  for (int64_t row0 = (static_cast<int64_t>(blockIdx.x) * kGateWarps + (threadIdx.x >> 5)) * kGateRows;
       row0 < rows; row0 += stride) {
    float o[kGateRows][VPL], z[kGateRows][VPL];
#pragma unroll
    for (int k = 0; k < kGateRows; ++k) {
      const int64_t row = row0 + k;
      if (row >= rows) break;
      IO::load_bf16(static_cast<const uint16_t*>(a.gate_z) + row * DV, lane, z[k]);
      if (a.out_f32) IO::load_f32(static_cast<const float*>(a.out) + row * DV, lane, o[k]);
      else IO::load_bf16(static_cast<const uint16_t*>(a.out) + row * DV, lane, o[k]);
    }
#pragma unroll
    for (int k = 0; k < kGateRows; ++k) {
      const int64_t row = row0 + k;
      if (row >= rows) break;
      float ss = 0.0f;
#pragma unroll
      for (int e = 0; e < VPL; ++e) ss = fmaf(o[k][e], o[k][e], ss);
      ss = warp_sum(ss);
      const float den = __fadd_rn(__fdiv_rn(ss, static_cast<float>(DV)), a.gate_eps);
      const float inv = den > 0.0f ? 1.0f / sqrtf(den) : 0.0f;  // all-zero row, eps 0
      float y[VPL];
#pragma unroll
      for (int e = 0; e < VPL; ++e) {
        const float act = a.gate_act == GDN_ACT_SIGMOID
                              ? __fdividef(1.0f, 1.0f + __expf(-z[k][e]))
                              : silu_fast(z[k][e]);
        y[e] = ((o[k][e] * inv) * w[e]) * act;
      }
      if (a.out_f32) IO::store_f32(static_cast<float*>(a.out) + row * DV, lane, y);
      else IO::store_bf16(static_cast<uint16_t*>(a.out) + row * DV, lane, y);
    }
  }
}

}  // namespace

cudaError_t launch_output_gate(const LayerArgs& a, int64_t rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t per_block = static_cast<int64_t>(kGateWarps) * kGateRows;
  const int64_t want = (rows + per_block - 1) / per_block;
  const int blocks = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
  switch (a.dv) {
    case 32: gate_rows_kernel<1><<<blocks, 32 * kGateWarps, 0, s>>>(a, rows); break;
    case 64: gate_rows_kernel<2><<<blocks, 32 * kGateWarps, 0, s>>>(a, rows); break;
    case 128: gate_rows_kernel<4><<<blocks, 32 * kGateWarps, 0, s>>>(a, rows); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gdn
