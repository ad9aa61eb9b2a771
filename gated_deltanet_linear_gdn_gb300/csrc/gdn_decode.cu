// gdn_decode.cu -- fused GDN decode step: conv roll + conv + SiLU, q|k|v
// split, QK L2 norm, fused gates and the gated delta rule, in one kernel.
//
// Sources: RL-Kernel PR #469 "C6: GDN decode-step goldens and recurrent/conv
// state contract", Summary (gating, QK norm x / sqrt(sum(x*x) + 1e-6) with
// scale on q after the norm, i_h = i_hv // (HV // H), state [num_blocks, HV,
// V, K]) and Notes "State ABI" (slots <= 0 skipped). The rule per value head:
//   S <- a S;  d = b (v - S k);  S <- S + d k^T;  o = S q.
//
// Design (HBM-bound: 4 MB of the ~4.3 MB per Qwen3-Next row is fp32 state).
// A work unit is (row, k-head): the Hv/Hk value heads of one k-head, whose
// states are one contiguous block of the pool and whose q, k and v conv
// channels belong to that unit alone (so the conv window is rolled by its only
// reader). The kernel is persistent -- one CTA per SM walks the units
// c, c + G, c + 2G, ... -- and warp-specialised:
//  - producer warp: streams each unit's state through a ring of shared-memory
//    stages (32 rows each) with bulk copies (cp.async.bulk, the TMA engine),
//    one "full" mbarrier per stage; it runs up to a ring's worth of stages
//    (192 KB) ahead, so in-flight bytes cost no registers;
//  - setup warps (one 8-channel conv group per thread): for the NEXT unit,
//    compute the conv (rolling its window), the L2-normalised q and k, k.q
//    and the gates into one of two buffers -- enough of them that this work
//    stays shorter than streaming a unit's state;
//  - 8 consumer warps: each takes 4 rows of every stage; a lane holds dk/32
//    consecutive floats of a row; S k and S q (before the update) share one
//    xor-shuffle butterfly, the read-out uses o = a (S q) + d (k . q) (equal to
//    (a S + d k^T) q), and the new rows go from registers to global memory with
//    128-bit streaming stores. Releasing a stage re-arms it for the producer.
// Every row's arithmetic is the same whatever unit order or CTA runs it, so
// results are bitwise independent of the batch composition. Every wait is
// bounded (GDN_DEVERR_TIMEOUT on expiry; the waiting role stops).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"

namespace gdn {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kStageRows = 32;
constexpr int kRowsPerWarp = kStageRows / kConsumerWarps;  // 4
constexpr int kRingBytes = 192 * 1024;

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

template <int DK, int R>
struct DecodeCfg {
  static constexpr int DV = DK;
  static constexpr int kUnitRows = R * DV;
  static constexpr int kStagesPerUnit = kUnitRows / kStageRows;
  static constexpr int kStageBytes = kStageRows * DK * 4;
  static constexpr int kNumStages = kRingBytes / kStageBytes;
  static constexpr int kGroups = (2 * DK + kUnitRows) / 8;  // 8-channel conv groups per unit
  static constexpr int kSetupWarps = (kGroups + 31) / 32 < 4 ? (kGroups + 31) / 32 : 4;
  static constexpr int kThreads = 32 * (1 + kSetupWarps + kConsumerWarps);
  static constexpr int kSetupFloats = 2 * DK + kUnitRows + 2 * R + 1;  // q^, k^, v, a, b, k.q
  static constexpr int kSetupStride = (kSetupFloats + 31) / 32 * 32;
  // dynamic shared memory: ring, two setup buffers, then the mbarriers
  static constexpr int kBarOffset = kRingBytes + 2 * kSetupStride * 4;
  static constexpr int kNumBars = 2 * kNumStages + 4;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8;
};

__device__ __forceinline__ bool unit_active(int32_t s, int num_slots) {
  return s > 0 && s < num_slots;
}

__device__ __forceinline__ void setup_barrier(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int DK, int R, bool kF32Cache>
__global__ void __launch_bounds__(DecodeCfg<DK, R>::kThreads, 1)
    decode_kernel(LayerArgs a, int num_units) {
  using Cfg = DecodeCfg<DK, R>;
  constexpr int DV = Cfg::DV;
  constexpr int VPL = DK / 32;
  constexpr int NS = Cfg::kNumStages;
  constexpr int SW = Cfg::kSetupWarps;
  using V = typename VecF<VPL>::T;

  extern __shared__ __align__(1024) unsigned char smem[];
  float* ring = reinterpret_cast<float*>(smem);
  float* setup = reinterpret_cast<float*>(smem + kRingBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOffset);
  // bars: full[NS], empty[NS], setup_full[2], setup_empty[2]
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NS);
  const uint32_t sfull0 = smem_addr(bars + 2 * NS), sempty0 = smem_addr(bars + 2 * NS + 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sfull0 + 8 * i, 32 * SW);
      mbar_init(sempty0 + 8 * i, kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int G = gridDim.x;
  const int per_unit_rows = Cfg::kUnitRows;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t g = 0;  // stages issued so far
      for (int u = blockIdx.x; u < num_units; u += G) {
        const int b = u / a.Hk, kh = u % a.Hk;
        const int32_t s = a.slot[b];
        if (!unit_active(s, a.num_slots)) continue;
        const float* src = a.ssm + (static_cast<int64_t>(s) * a.Hv + kh * R) * (DV * DK);
        bool ok = true;
        for (int k = 0; k < Cfg::kStagesPerUnit; ++k, ++g) {
          const uint32_t r = g % NS, c = g / NS;
          if (!mbar_wait_bounded(empty0 + 8 * r, (c & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(full0 + 8 * r, Cfg::kStageBytes);
          bulk_g2s(smem_addr(ring + static_cast<size_t>(r) * kStageRows * DK),
                   src + static_cast<int64_t>(k) * kStageRows * DK, Cfg::kStageBytes, full0 + 8 * r);
        }
        if (!ok) {
          if (a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
          break;
        }
      }
    }
    return;
  }

  if (warp >= 1 && warp <= SW) {
    // ------------------------------------------------------------ setup
    // SW warps, one 8-channel conv group per thread; they meet at a named
    // barrier, then warp 1 normalises q and k and computes k.q and the gates.
    // Every setup thread passes every barrier even after a timeout, so none
    // can be left waiting on a named barrier.
    constexpr int QG = DK / 8;
    constexpr int NG = Cfg::kGroups;
    const int st = tid - 32;  // 0 .. 32*SW-1
    bool failed = false;
    uint32_t n = 0;  // active units prepared so far
    for (int u = blockIdx.x; u < num_units; u += G) {
      const int b = u / a.Hk, kh = u % a.Hk;
      const int32_t s = a.slot[b];
      if (!unit_active(s, a.num_slots)) {
        if (s >= a.num_slots && st == 0 && kh == 0 && a.err) atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
        continue;
      }
      const uint32_t p = n & 1, use = n >> 1;
      if (!failed && !mbar_wait_bounded(sempty0 + 8 * p, (use & 1) ^ 1)) {
        if (a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
        failed = true;
      }
      float* buf = setup + p * Cfg::kSetupStride;
      float* qb = buf;
      float* kb = buf + DK;
      float* vb = buf + 2 * DK;
      float* gb = buf + 2 * DK + Cfg::kUnitRows;  // a[R], b[R], k.q
      if (!failed) {
        const uint16_t* xrow = static_cast<const uint16_t*>(a.mixed) + static_cast<int64_t>(b) * a.D;
        for (int g = st; g < NG; g += 32 * SW) {
          int c0;
          float* dst;
          if (g < QG) { c0 = kh * DK + 8 * g; dst = qb + 8 * g; }
          else if (g < 2 * QG) { c0 = (a.Hk + kh) * DK + 8 * (g - QG); dst = kb + 8 * (g - QG); }
          else { c0 = 2 * a.Hk * DK + kh * R * DV + 8 * (g - 2 * QG); dst = vb + 8 * (g - 2 * QG); }
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
      if (SW > 1) setup_barrier(32 * SW);
      else __syncwarp();
      if (warp == 1 && !failed) {
        float qv[VPL], kv[VPL], sq = 0.0f, sk = 0.0f;
#pragma unroll
        for (int e = 0; e < VPL; ++e) {
          qv[e] = qb[lane * VPL + e];
          kv[e] = kb[lane * VPL + e];
          sq = fmaf(qv[e], qv[e], sq);
          sk = fmaf(kv[e], kv[e], sk);
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float iq = a.qk_l2norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
        const float ik = a.qk_l2norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
        float kq = 0.0f;
#pragma unroll
        for (int e = 0; e < VPL; ++e) {
          qv[e] = (qv[e] * iq) * a.scale;
          kv[e] = kv[e] * ik;
          kq = fmaf(kv[e], qv[e], kq);
        }
        kq = warp_sum(kq);
#pragma unroll
        for (int e = 0; e < VPL; ++e) {
          qb[lane * VPL + e] = qv[e];
          kb[lane * VPL + e] = kv[e];
        }
        if (lane < R) {
          const int h = kh * R + lane;
          float al, be;
          gate_values(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                      static_cast<int64_t>(b) * a.Hv + h, h, al, be);
          gb[lane] = al;
          gb[R + lane] = be;
        }
        if (lane == 0) gb[2 * R] = kq;
      }
      mbar_arrive(sfull0 + 8 * p);  // every setup thread: its writes are released
      ++n;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1 - SW;
  uint32_t g = 0, n = 0;
  for (int u = blockIdx.x; u < num_units; u += G) {
    const int b = u / a.Hk, kh = u % a.Hk;
    const int32_t s = a.slot[b];
    const int64_t out_base = (static_cast<int64_t>(b) * a.Hv + kh * R) * DV;
    if (!unit_active(s, a.num_slots)) {  // inactive / invalid row: zero outputs, no state touched
      for (int i = cw * 32 + lane; i < per_unit_rows; i += kConsumerWarps * 32) {
        if (a.out_f32) static_cast<float*>(a.out)[out_base + i] = 0.0f;
        else static_cast<uint16_t*>(a.out)[out_base + i] = 0;
      }
      continue;
    }
    const uint32_t p = n & 1;
    if (!mbar_wait_bounded(sfull0 + 8 * p, (n >> 1) & 1)) {
      if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
      return;
    }
    const float* buf = setup + p * Cfg::kSetupStride;
    float qv[VPL], kv[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
      qv[e] = buf[lane * VPL + e];
      kv[e] = buf[DK + lane * VPL + e];
    }
    const float* vb = buf + 2 * DK;
    const float* gb = buf + 2 * DK + per_unit_rows;
    const float kq = gb[2 * R];
    float* dst_base = a.ssm + (static_cast<int64_t>(s) * a.Hv + kh * R) * (DV * DK);
    for (int k = 0; k < Cfg::kStagesPerUnit; ++k, ++g) {
      const uint32_t r = g % NS, c = g / NS;
      if (!mbar_wait_bounded(full0 + 8 * r, c & 1)) {
        if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
        return;
      }
      const int row0 = k * kStageRows + cw * kRowsPerWarp;
      const int hl = row0 / DV;
      const float al = gb[hl], be = gb[R + hl];
      const float* src = ring + static_cast<size_t>(r) * kStageRows * DK + cw * kRowsPerWarp * DK;
      float o[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        float sv[VPL];
        vec_to<VPL>(reinterpret_cast<const V*>(src + i * DK)[lane], sv);
        float pk = 0.0f, pq = 0.0f;
#pragma unroll
        for (int e = 0; e < VPL; ++e) { pk = fmaf(sv[e], kv[e], pk); pq = fmaf(sv[e], qv[e], pq); }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          pk += __shfl_xor_sync(0xffffffffu, pk, off);
          pq += __shfl_xor_sync(0xffffffffu, pq, off);
        }
        const float delta = be * (vb[row0 + i] - al * pk);
        float nw[VPL];
#pragma unroll
        for (int e = 0; e < VPL; ++e) nw[e] = fmaf(delta, kv[e], al * sv[e]);
        __stcs(reinterpret_cast<V*>(dst_base + static_cast<int64_t>(row0 + i) * DK) + lane,
               vec_from<VPL>(nw));
        o[i] = fmaf(delta, kq, al * pq);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * r);  // this warp is done with the stage
      if (lane < kRowsPerWarp) {
        float ov = o[0];
#pragma unroll
        for (int i = 1; i < kRowsPerWarp; ++i) ov = (lane == i) ? o[i] : ov;
        if (a.out_f32) static_cast<float*>(a.out)[out_base + row0 + lane] = ov;
        else static_cast<uint16_t*>(a.out)[out_base + row0 + lane] = f2bf(ov);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sempty0 + 8 * p);  // this warp no longer reads the setup buffer
    ++n;
  }
}

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (count[dev] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
      c = 148;
    count[dev] = c;
  }
  return count[dev];
}

template <int DK, int R, bool kF32Cache>
cudaError_t launch_one(const LayerArgs& a, int B, cudaStream_t s) {
  using Cfg = DecodeCfg<DK, R>;
  auto kern = decode_kernel<DK, R, kF32Cache>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int units = B * a.Hk;
  const int grid = units < sm_count() ? units : sm_count();
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, s>>>(a, units);
  return cudaGetLastError();
}

template <int DK, int R>
cudaError_t launch_dk_r(const LayerArgs& a, int B, cudaStream_t s) {
  if (a.conv_f32) return launch_one<DK, R, true>(a, B, s);
  return launch_one<DK, R, false>(a, B, s);
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
