// gdn_decode.cu -- fused GDN decode step: conv roll + conv + SiLU, q|k|v
// split, QK L2 norm, fused gates and the gated delta rule, in one kernel.
//
// Sources: RL-Kernel PR #469 "C6: GDN decode-step goldens and recurrent/conv
// state contract", Summary (gating, QK norm x / sqrt(sum(x*x) + 1e-6) with
// scale on q after the norm, i_h = i_hv // (HV // H), state [num_blocks, HV,
// V, K]) and Notes "State ABI" (slots <= 0 skipped). The rule per value head:
//   S <- a S;  d = b (v - S k);  S <- S + d k^T;  o = S q.
//
// Design (HBM-bound: 4 MB of the ~4.3 MB per Qwen3-Next row is fp32 state):
//  - one CTA per (row, k-head). Its Hv/Hk value heads are consecutive in the
//    state pool, so the CTA streams ONE contiguous block of R*dv*dk floats,
//    and it alone rolls the conv channels of its q, k and v heads.
//  - state rows (one dv index, dk floats) are independent: a warp owns a run
//    of rows; a lane holds dk/32 consecutive floats of a row (128-bit loads
//    for dk = 128), so a warp instruction moves one 512-byte row.
//  - both dot products a row needs (S k and S q, before the update) share one
//    xor-shuffle butterfly; the read-out uses o = a (S q) + d (k . q), which
//    equals (a S + d k^T) q.
//  - the first batch of state rows is requested before the conv phase, and
//    each batch's loads are issued before the previous batch is consumed.
//  - no block-wide reduction reuses shared storage: the two norm reductions
//    are single-warp shuffles into distinct shared slots, read after a barrier.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

template <int N> struct VecF;
template <> struct VecF<1> { using T = float; };
template <> struct VecF<2> { using T = float2; };
template <> struct VecF<4> { using T = float4; };

template <int N>
__device__ __forceinline__ void vec_to(const typename VecF<N>::T& v, float (&f)[N]);
template <> __device__ __forceinline__ void vec_to<1>(const float& v, float (&f)[1]) { f[0] = v; }
template <> __device__ __forceinline__ void vec_to<2>(const float2& v, float (&f)[2]) { f[0] = v.x; f[1] = v.y; }
template <> __device__ __forceinline__ void vec_to<4>(const float4& v, float (&f)[4]) {
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <int N>
__device__ __forceinline__ typename VecF<N>::T vec_from(const float (&f)[N]);
template <> __device__ __forceinline__ float vec_from<1>(const float (&f)[1]) { return f[0]; }
template <> __device__ __forceinline__ float2 vec_from<2>(const float (&f)[2]) { return make_float2(f[0], f[1]); }
template <> __device__ __forceinline__ float4 vec_from<4>(const float (&f)[4]) {
  return make_float4(f[0], f[1], f[2], f[3]);
}

template <int DK, int R, bool kF32Cache>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(LayerArgs a) {
  constexpr int DV = DK;
  constexpr int ROWS = R * DV;            // state rows owned by this CTA
  constexpr int RPW = ROWS / kDecWarps;   // rows per warp
  constexpr int VPL = DK / 32;            // floats of a row per lane
  constexpr int NB = 4;                   // rows per batch
  constexpr int NBATCH = RPW / NB;
  static_assert(RPW % NB == 0, "rows per warp must be a multiple of the batch");
  using V = typename VecF<VPL>::T;

  __shared__ float q_s[DK], k_s[DK], v_s[ROWS], o_s[ROWS];
  __shared__ float alpha_s[R], beta_s[R], inv_s[2];

  const int kh = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hv0 = kh * R;
  const int64_t out_base = (static_cast<int64_t>(b) * a.Hv + hv0) * DV;
  const int32_t s = a.slot[b];

  if (s <= 0 || s >= a.num_slots) {  // inactive or invalid row: zero output, no state touched
    if (s >= a.num_slots && tid == 0 && a.err) atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
    for (int i = tid; i < ROWS; i += kDecThreads) {
      if (a.out_f32) static_cast<float*>(a.out)[out_base + i] = 0.0f;
      else static_cast<uint16_t*>(a.out)[out_base + i] = 0;
    }
    return;
  }

  float* S = a.ssm + (static_cast<int64_t>(s) * a.Hv + hv0) * (DV * DK);
  const int row0 = warp * RPW;
  V cur[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i)
    cur[i] = __ldcs(reinterpret_cast<const V*>(S + static_cast<int64_t>(row0 + i) * DK) + lane);

  // ---- conv (or bypass) of this CTA's q, k and v channels -> shared ----
  {
    constexpr int QG = DK / 8, NG = (2 * DK + ROWS) / 8;
    const uint16_t* xrow = static_cast<const uint16_t*>(a.mixed) + static_cast<int64_t>(b) * a.D;
    for (int g = tid; g < NG; g += kDecThreads) {
      int c0;
      float* dst;
      if (g < QG) { c0 = kh * DK + 8 * g; dst = q_s + 8 * g; }
      else if (g < 2 * QG) { c0 = (a.Hk + kh) * DK + 8 * (g - QG); dst = k_s + 8 * (g - QG); }
      else { c0 = 2 * a.Hk * DK + hv0 * DV + 8 * (g - 2 * QG); dst = v_s + 8 * (g - 2 * QG); }
      float x8[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(xrow + c0)), x8);
      if (a.conv_w) {
        float win[8][kConvW - 1], y8[8];
        load_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, win);
        conv8_step<kF32Cache>(win, x8, static_cast<const uint16_t*>(a.conv_w),
                              static_cast<const uint16_t*>(a.conv_b), c0, a.silu != 0, y8);
        store_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, win);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = y8[i];
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = x8[i];
      }
    }
  }
  __syncthreads();

  // ---- norms (one warp each) and gates ----
  if (warp < 2) {
    const float* src = warp == 0 ? q_s : k_s;
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < VPL; ++e) { const float x = src[lane * VPL + e]; ss = fmaf(x, x, ss); }
    ss = warp_sum(ss);
    if (lane == 0) inv_s[warp] = a.qk_l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
  } else if (warp == 2 && lane < R) {
    const int h = hv0 + lane;
    float al, be;
    gate_values(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias, static_cast<int64_t>(b) * a.Hv + h, h,
                al, be);
    alpha_s[lane] = al;
    beta_s[lane] = be;
  }
  __syncthreads();

  float qv[VPL], kv[VPL];
  {
    const float iq = inv_s[0], ik = inv_s[1];
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
      qv[e] = (q_s[lane * VPL + e] * iq) * a.scale;
      kv[e] = k_s[lane * VPL + e] * ik;
    }
  }
  float kq = 0.0f;
#pragma unroll
  for (int e = 0; e < VPL; ++e) kq = fmaf(kv[e], qv[e], kq);
  kq = warp_sum(kq);

  // ---- stream the state rows ----
#pragma unroll
  for (int bt = 0; bt < NBATCH; ++bt) {
    V nxt[NB];
    if (bt + 1 < NBATCH) {
#pragma unroll
      for (int i = 0; i < NB; ++i)
        nxt[i] = __ldcs(reinterpret_cast<const V*>(S + static_cast<int64_t>(row0 + (bt + 1) * NB + i) * DK) + lane);
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int row = row0 + bt * NB + i;
      const int hl = row / DV;
      float sv[VPL];
      vec_to<VPL>(cur[i], sv);
      float pk = 0.0f, pq = 0.0f;
#pragma unroll
      for (int e = 0; e < VPL; ++e) { pk = fmaf(sv[e], kv[e], pk); pq = fmaf(sv[e], qv[e], pq); }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        pk += __shfl_xor_sync(0xffffffffu, pk, o);
        pq += __shfl_xor_sync(0xffffffffu, pq, o);
      }
      const float al = alpha_s[hl], be = beta_s[hl];
      const float delta = be * (v_s[row] - al * pk);
      float nw[VPL];
#pragma unroll
      for (int e = 0; e < VPL; ++e) nw[e] = fmaf(delta, kv[e], al * sv[e]);
      __stcs(reinterpret_cast<V*>(S + static_cast<int64_t>(row) * DK) + lane, vec_from<VPL>(nw));
      if (lane == 0) o_s[row] = fmaf(delta, kq, al * pq);
    }
    if (bt + 1 < NBATCH) {
#pragma unroll
      for (int i = 0; i < NB; ++i) cur[i] = nxt[i];
    }
  }
  __syncwarp();
  for (int r = lane; r < RPW; r += 32) {
    const float o = o_s[row0 + r];
    if (a.out_f32) static_cast<float*>(a.out)[out_base + row0 + r] = o;
    else static_cast<uint16_t*>(a.out)[out_base + row0 + r] = f2bf(o);
  }
}

template <int DK, int R>
cudaError_t launch_dk_r(const LayerArgs& a, int B, cudaStream_t s) {
  dim3 grid(a.Hk, B);
  if (a.conv_f32) decode_kernel<DK, R, true><<<grid, kDecThreads, 0, s>>>(a);
  else decode_kernel<DK, R, false><<<grid, kDecThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const LayerArgs& a, int B, cudaStream_t s) {
  switch (a.Hv / a.Hk) {
    case 1: return launch_dk_r<DK, 1>(a, B, s);
    case 2: return launch_dk_r<DK, 2>(a, B, s);
    case 4: return launch_dk_r<DK, 4>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const LayerArgs& a, int B, cudaStream_t s) {
  switch (a.dk) {
    case 32: return launch_dk<32>(a, B, s);
    case 64: return launch_dk<64>(a, B, s);
    case 128: return launch_dk<128>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
