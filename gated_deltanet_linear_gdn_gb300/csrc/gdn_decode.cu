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
//    stages (64 rows each) with bulk copies (cp.async.bulk, the TMA engine),
//    one "full" mbarrier per stage; it runs up to a ring's worth of stages
//    (192 KB) ahead, so in-flight bytes cost no registers;
//  - 2 setup warps: per unit, the conv (rolling its windows), the
//    L2-normalised q and k, k.q and the gates, written to a setup buffer; every
//    global load of a unit (gate inputs, input channels, conv windows and
//    parameters) is issued before anything waits on it. Two schemes, chosen by
//    measurement: with an fp32 state the warps share each unit (one conv group
//    per thread, a named barrier, two buffers) -- the shortest setup per unit;
//    with a bf16 state, whose units stream in half the time, each warp
//    prepares whole units (unit n to warp n % 2, buffer n % 4) so that two are
//    in flight;
//  - 8 consumer warps: each loads its 8 rows of a stage into registers (a lane
//    holds dk/32 consecutive elements of a row) and hands the stage straight
//    back to the producer. The 16 dot products (S k and S q before the update,
//    per row) are summed in one transposed butterfly -- 15 exchanges that halve
//    the values each lane holds, then one plain step -- instead of 16 separate
//    5-step butterflies; a lane pair then holds both dots of its row, computes
//    d = b (v - a S k) and o = a (S q) + d (k . q) (equal to (a S + d k^T) q),
//    and the d's are broadcast for the row updates (packed f32x2 arithmetic),
//    which go from registers to global memory with streaming stores.
// The state may be stored as fp32 or bf16 (the arithmetic is fp32 either way; a
// bf16 store rounds to nearest even), which halves the bytes a step moves.
// Every row's arithmetic is the same whatever unit order or CTA runs it, so
// results are bitwise independent of the batch composition. Every wait is
// bounded (GDN_DEVERR_TIMEOUT on expiry; the waiting role stops).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"

namespace gdn {

namespace {

constexpr int kConsumerWarps = 8;

// Test hook (gdn_testing_set_fault, mode 1): the first consumer warp of CTA 0 waits, with a
// 10 ms bound, on a barrier nothing arrives on, and leaves as a consumer whose wait ran out
// does, so that the kernel's bounded waits and error reporting run on the GPU. 0 in use.
__device__ int g_test_fault = 0;
constexpr uint64_t kTestWaitNs = 10000000ull;
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

// One lane's VPL consecutive state elements of a row: fp32 in registers, stored as
// fp32 or (bf16 state) bf16 rounded to nearest even.
template <int VPL, bool kBf16State>
struct StateIO;
template <int VPL>
struct StateIO<VPL, false> {
  __device__ static void load(const void* row, int lane, float (&v)[VPL]) {
    vec_to<VPL>(reinterpret_cast<const typename VecF<VPL>::T*>(row)[lane], v);
  }
  __device__ static void store(void* row, int lane, const float (&v)[VPL]) {
    __stcs(reinterpret_cast<typename VecF<VPL>::T*>(row) + lane, vec_from<VPL>(v));
  }
};
template <>
struct StateIO<4, true> {
  __device__ static void load(const void* row, int lane, float (&v)[4]) {
    const uint2 u = reinterpret_cast<const uint2*>(row)[lane];
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
  }
  __device__ static void store(void* row, int lane, const float (&v)[4]) {
    uint2 u;
    u.x = pack_bf2(v[0], v[1]);
    u.y = pack_bf2(v[2], v[3]);
    __stcs(reinterpret_cast<uint2*>(row) + lane, u);
  }
};
template <>
struct StateIO<2, true> {
  __device__ static void load(const void* row, int lane, float (&v)[2]) {
    const uint32_t u = reinterpret_cast<const uint32_t*>(row)[lane];
    v[0] = __uint_as_float(u << 16); v[1] = __uint_as_float(u & 0xFFFF0000u);
  }
  __device__ static void store(void* row, int lane, const float (&v)[2]) {
    __stcs(reinterpret_cast<unsigned int*>(row) + lane, pack_bf2(v[0], v[1]));
  }
};
template <>
struct StateIO<1, true> {
  __device__ static void load(const void* row, int lane, float (&v)[1]) {
    v[0] = bf2f(reinterpret_cast<const uint16_t*>(row)[lane]);
  }
  __device__ static void store(void* row, int lane, const float (&v)[1]) {
    reinterpret_cast<uint16_t*>(row)[lane] = f2bf(v[0]);
  }
};

// A lane's share of a row dot product and of the row update, in packed f32x2
// arithmetic where the lane holds an even number of elements.
template <int VPL>
__device__ __forceinline__ float lane_dot(const float (&s)[VPL], const float (&x)[VPL]) {
  if constexpr (VPL == 1) {
    return __fmul_rn(s[0], x[0]);
  } else {
    float2 acc = __fmul2_rn(make_float2(s[0], s[1]), make_float2(x[0], x[1]));
#pragma unroll
    for (int e = 2; e < VPL; e += 2)
      acc = __ffma2_rn(make_float2(s[e], s[e + 1]), make_float2(x[e], x[e + 1]), acc);
    return acc.x + acc.y;
  }
}
// s <- al s + d k (each element: fma(d, k, al * s)).
template <int VPL>
__device__ __forceinline__ void lane_update(float (&s)[VPL], const float (&k)[VPL], float al,
                                            float d) {
  if constexpr (VPL == 1) {
    s[0] = fmaf(d, k[0], al * s[0]);
  } else {
#pragma unroll
    for (int e = 0; e < VPL; e += 2) {
      const float2 r = __ffma2_rn(make_float2(d, d), make_float2(k[e], k[e + 1]),
                                  __fmul2_rn(make_float2(al, al), make_float2(s[e], s[e + 1])));
      s[e] = r.x;
      s[e + 1] = r.y;
    }
  }
}

// Sums V per-lane values across the warp, V in {8, 16}: V-1 exchanges halve the
// values a lane holds (at each level a lane keeps the half selected by its lane
// bit and adds the partner's copy of it), then plain butterflies finish. On return
// red[0] of lane L is the full sum of value L / (32 / V).
template <int V>
__device__ __forceinline__ void transposed_warp_sum(float (&red)[V], int lane) {
  constexpr int LPV = 32 / V;
#pragma unroll
  for (int lvl = 0; (1 << lvl) < V; ++lvl) {
    const int m = 16 >> lvl;
    const int h = V >> (lvl + 1);
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < h; ++j) {
      const float keep = up ? red[h + j] : red[j];
      const float give = up ? red[j] : red[h + j];
      red[j] = keep + __shfl_xor_sync(0xffffffffu, give, m);
    }
  }
#pragma unroll
  for (int m = LPV / 2; m >= 1; m >>= 1) red[0] += __shfl_xor_sync(0xffffffffu, red[0], m);
}

// The dot products of a warp's RPW state rows (held in sv, a lane owning VPL consecutive
// elements of each) with k and q, summed in one transposed butterfly; then for row
// ri = lane / (2 LPV): d = b (v - a (S k)) and o = a (S q) + d (k . q). Lanes with
// `writer` set hold the row's o. Both decode kernels run a row through this one function.
template <int VPL, int RPW>
__device__ __forceinline__ void rows_predict(const float (&sv)[RPW][VPL], const float (&qv)[VPL],
                                             const float (&kv)[VPL], const float* vb, int row0,
                                             float al, float be, float kq, int lane,
                                             float& delta, float& ov, int& ri, bool& writer) {
  float red[2 * RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    red[2 * i] = lane_dot<VPL>(sv[i], kv);
    red[2 * i + 1] = lane_dot<VPL>(sv[i], qv);
  }
  transposed_warp_sum<2 * RPW>(red, lane);
  // lanes of value pair i (row i) swap halves: both then hold (S k)_i and (S q)_i
  constexpr int LPV = 32 / (2 * RPW);
  const float other = __shfl_xor_sync(0xffffffffu, red[0], LPV);
  const bool is_q = ((lane / LPV) & 1) != 0;
  const float pk = is_q ? other : red[0], pq = is_q ? red[0] : other;
  ri = lane / (2 * LPV);
  // explicit roundings: no compiled copy of this code may contract it differently
  delta = __fmul_rn(be, __fmaf_rn(-al, pk, vb[row0 + ri]));
  writer = lane % (2 * LPV) == 0;
  ov = __fmaf_rn(delta, kq, __fmul_rn(al, pq));  // o_i = a (S q)_i + d_i (k . q)
}

// The warp's rows after the predict step: S <- a S + d k^T row by row (d of row i from the
// lanes that computed it), each stored as soon as it is updated.
template <int VPL, int RPW, bool kBf16State>
__device__ __forceinline__ void rows_update_store(float (&sv)[RPW][VPL], const float (&kv)[VPL],
                                                  float al, float delta, unsigned char* dst,
                                                  int row_bytes, int lane) {
  constexpr int LPV = 32 / (2 * RPW);
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const float d = __shfl_sync(0xffffffffu, delta, i * 2 * LPV);
    lane_update<VPL>(sv[i], kv, al, d);
    StateIO<VPL, kBf16State>::store(dst + static_cast<int64_t>(i) * row_bytes, lane, sv[i]);
  }
}

template <int DK, int R, bool kBf16State>
struct DecodeCfg {
  static constexpr int DV = DK;
  static constexpr int kElemBytes = kBf16State ? 2 : 4;
  static constexpr int kRowBytes = DK * kElemBytes;
  static constexpr int kUnitRows = R * DV;
  // 64-row stages (8 rows per consumer warp), or the whole unit when it is smaller
  static constexpr int kStageRows = kUnitRows < 64 ? kUnitRows : 64;
  static constexpr int kRowsPerWarp = kStageRows / kConsumerWarps;
  static constexpr int kStagesPerUnit = kUnitRows / kStageRows;
  static constexpr int kStageBytes = kStageRows * kRowBytes;
  static_assert(kUnitRows % kStageRows == 0 && DV % kRowsPerWarp == 0, "stage tiling");
  static_assert(kRowsPerWarp == 4 || kRowsPerWarp == 8, "the reduction handles 8 or 16 values");
  // Setup scheme (both measured): with an fp32 state the setup warps share each
  // unit (shortest time per unit; two buffers); with a bf16 state, whose units
  // stream in half the time, each warp prepares whole units so that two are in
  // flight (four buffers).
  static constexpr bool kCoopSetup = !kBf16State;
  static constexpr int kNumStages = kRingBytes / kStageBytes;
  static constexpr int kGroups = (2 * DK + kUnitRows) / 8;  // 8-channel conv groups per unit
  static constexpr int kSetupWarps = 2;
  static constexpr int kSetupBufs = kCoopSetup ? 2 : 2 * kSetupWarps;
  // + 1 epilogue warp (the output gate; it returns at once in an ungated call)
  static constexpr int kEpiWarp = 1 + kSetupWarps + kConsumerWarps;
  static constexpr int kThreads = 32 * (kEpiWarp + 1);
  static constexpr int kSetupFloats = 2 * DK + kUnitRows + 2 * R + 1;  // q^, k^, v, a, b, k.q
  static constexpr int kSetupStride = (kSetupFloats + 31) / 32 * 32;
  // dynamic shared memory: ring, the setup buffers, two unit-sized o buffers
  // (gated calls), then the mbarriers
  static constexpr int kOBufOffset = kRingBytes + kSetupBufs * kSetupStride * 4;
  static constexpr int kBarOffset = kOBufOffset + 2 * kUnitRows * 4;
  static constexpr int kNumBars = 2 * kNumStages + 2 * kSetupBufs + 5;  // + the test hook's
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8;
  static_assert(kSmemBytes <= 227 * 1024, "decode shared memory exceeds the per-CTA limit");
};

// Conv group g (8 channels) of unit (row b, k-head kh): its first channel in the
// packed q|k|v vector and its slot in the setup buffer (q^, k^, v).
template <int DK, int R>
__device__ __forceinline__ void group_channels(int g, int kh, int Hk, float* buf, int& c0,
                                               float*& dst) {
  constexpr int QG = DK / 8;
  if (g < QG) { c0 = kh * DK + 8 * g; dst = buf + 8 * g; }
  else if (g < 2 * QG) { c0 = (Hk + kh) * DK + 8 * (g - QG); dst = buf + DK + 8 * (g - QG); }
  else { c0 = 2 * Hk * DK + kh * R * DK + 8 * (g - 2 * QG); dst = buf + 2 * DK + 8 * (g - 2 * QG); }
}

// Every global load of one conv group: the input channels, the conv window and
// the conv parameters (issued together, before anything waits on them).
template <bool kF32Cache>
struct GroupLoads {
  uint4 x;
  RawWin8<kF32Cache> win;
  ConvParams8 prm;
};
template <bool kF32Cache>
__device__ __forceinline__ void group_load(const LayerArgs& a, const uint16_t* xrow, int32_t s,
                                           int c0, GroupLoads<kF32Cache>& L) {
  L.x = __ldg(reinterpret_cast<const uint4*>(xrow + c0));
  if (a.conv_w) {
    load_conv8_raw<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, L.win);
    L.prm = conv8_params(static_cast<const uint16_t*>(a.conv_w),
                         static_cast<const uint16_t*>(a.conv_b), c0);
  }
}
// The group's conv (rolling and storing its window) into dst[0..8).
template <bool kF32Cache>
__device__ __forceinline__ void group_conv(const LayerArgs& a, int32_t s, int c0,
                                           const GroupLoads<kF32Cache>& L, float* dst) {
  float x8[8];
  unpack8(L.x, x8);
  if (a.conv_w) {
    float win[8][kConvW - 1], y8[8];
    unpack_conv8<kF32Cache>(L.win, a.conv_layout, win);
    conv8_apply<kF32Cache>(win, x8, L.prm, a.silu != 0, y8);
    store_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, win);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = y8[i];
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = x8[i];
  }
}

// One warp, after the conv outputs are in the buffer: L2-normalise q (then scale)
// and k in place, k.q and the gates of the unit's R heads (raw inputs in lanes < R).
template <int DK, int R>
__device__ __forceinline__ void finish_setup(const LayerArgs& a, float* buf, const GateRaw& gr,
                                             int lane) {
  constexpr int VPL = DK / 32;
  float* qb = buf;
  float* kb = buf + DK;
  float* gb = buf + 2 * DK + R * DK;  // a[R], b[R], k.q
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
  __syncwarp();
#pragma unroll
  for (int e = 0; e < VPL; ++e) {
    qb[lane * VPL + e] = qv[e];
    kb[lane * VPL + e] = kv[e];
  }
  if (lane < R) {
    float al, be;
    gate_from_raw(gr, a.gate_mode, al, be);
    gb[lane] = al;
    gb[R + lane] = be;
  }
  if (lane == 0) gb[2 * R] = kq;
}

__device__ __forceinline__ bool unit_active(int32_t s, int num_slots) {
  return s > 0 && s < num_slots;
}

__device__ __forceinline__ void setup_barrier(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// The slots of this CTA's units (unit i is blockIdx.x + i * gridDim.x) for one
// warp: read 32 units at a time (lane j holds unit i0 + j's slot) with the next
// 32 already in flight, and handed out by shuffle -- so walking the units costs no
// dependent global load per unit. Every lane of the warp must call get().
struct UnitSlots {
  int base = -64;
  int32_t cur = 0, nxt = 0;
  __device__ __forceinline__ int32_t load(const LayerArgs& a, int i0, int num_units, int lane) {
    const int u = blockIdx.x + (i0 + lane) * static_cast<int>(gridDim.x);
    return u < num_units ? a.slot[u / a.Hk] : 0;
  }
  __device__ __forceinline__ int32_t get(const LayerArgs& a, int i, int num_units, int lane) {
    const int b0 = i & ~31;
    if (b0 != base) {
      cur = (b0 == base + 32) ? nxt : load(a, b0, num_units, lane);
      base = b0;
      nxt = load(a, b0 + 32, num_units, lane);
    }
    return __shfl_sync(0xffffffffu, cur, i & 31);
  }
};

template <int DK, int R, bool kF32Cache, bool kBf16State>
__global__ void __launch_bounds__(DecodeCfg<DK, R, kBf16State>::kThreads, 1)
    decode_kernel(LayerArgs a, int num_units) {
  using Cfg = DecodeCfg<DK, R, kBf16State>;
  using IO = StateIO<DK / 32, kBf16State>;
  constexpr int DV = Cfg::DV;
  constexpr int VPL = DK / 32;
  constexpr int NS = Cfg::kNumStages;
  constexpr int SW = Cfg::kSetupWarps;
  constexpr int NB = Cfg::kSetupBufs;

  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* ring = smem;
  float* setup = reinterpret_cast<float*>(smem + kRingBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOffset);
  float* obuf = reinterpret_cast<float*>(smem + Cfg::kOBufOffset);
  // bars: full[NS], empty[NS], setup_full[NB], setup_empty[NB], o_full[2], o_empty[2]
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NS);
  const uint32_t sfull0 = smem_addr(bars + 2 * NS), sempty0 = smem_addr(bars + 2 * NS + NB);
  const uint32_t ofull0 = smem_addr(bars + 2 * NS + 2 * NB);
  const uint32_t oempty0 = smem_addr(bars + 2 * NS + 2 * NB + 2);
  const uint32_t dead = smem_addr(bars + 2 * NS + 2 * NB + 4);  // never arrived on

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kConsumerWarps);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(sfull0 + 8 * i, Cfg::kCoopSetup ? 32 * SW : 32);
      mbar_init(sempty0 + 8 * i, kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ofull0 + 8 * i, kConsumerWarps);
      mbar_init(oempty0 + 8 * i, 1);
    }
    mbar_init(dead, 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int G = gridDim.x;
  const int per_unit_rows = Cfg::kUnitRows;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The warp walks the units (for the slot batches); lane 0 issues the copies.
    UnitSlots slots;
    uint32_t g = 0;  // stages issued so far (lane 0)
    bool ok = true;
    for (int i = 0, u = blockIdx.x; u < num_units && ok; ++i, u += G) {
      const int kh = u % a.Hk;
      const int32_t s = slots.get(a, i, num_units, lane);
      if (!unit_active(s, a.num_slots)) continue;
      if (lane == 0) {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(a.ssm) +
                                   (static_cast<int64_t>(s) * a.Hv + kh * R) * (DV * Cfg::kRowBytes);
        for (int k = 0; k < Cfg::kStagesPerUnit; ++k, ++g) {
          const uint32_t r = g % NS, c = g / NS;
          if (!mbar_wait_bounded(empty0 + 8 * r, (c & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(full0 + 8 * r, Cfg::kStageBytes);
          bulk_g2s(smem_addr(ring + static_cast<size_t>(r) * Cfg::kStageBytes),
                   src + static_cast<int64_t>(k) * Cfg::kStageBytes, Cfg::kStageBytes, full0 + 8 * r);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (!ok && lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
    return;
  }

  if (warp >= 1 && warp <= SW) {
    // ------------------------------------------------------------ setup
    constexpr int NG = Cfg::kGroups;
    uint32_t n = 0;  // ordinal of the next active unit
    if constexpr (Cfg::kCoopSetup) {
      // The SW warps share each unit, one conv group per thread; they meet at a
      // named barrier, then the first setup warp normalises q and k and writes
      // k.q and the gates. This scheme waits for its buffer before loading and
      // loads the gate inputs last: with an fp32 state (HBM-saturated) that
      // measured faster than issuing the unit's loads early. Every setup thread
      // passes every barrier even after a timeout, so none is left waiting on
      // the named barrier.
      const int st = tid - 32;  // 0 .. 32*SW-1
      bool failed = false;
      for (int u = blockIdx.x; u < num_units; u += G) {
        const int b = u / a.Hk, kh = u % a.Hk;
        const int32_t s = a.slot[b];
        if (!unit_active(s, a.num_slots)) {
          if (s >= a.num_slots && st == 0 && kh == 0 && a.err) atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
          continue;
        }
        const uint32_t p = n % NB, use = n / NB;
        if (!failed && !mbar_wait_bounded(sempty0 + 8 * p, (use & 1) ^ 1)) {
          if (a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
          failed = true;
        }
        float* buf = setup + p * Cfg::kSetupStride;
        if (!failed) {
          const uint16_t* xrow = static_cast<const uint16_t*>(a.mixed) + static_cast<int64_t>(b) * a.D;
          for (int g = st; g < NG; g += 32 * SW) {
            int c0;
            float* dst;
            group_channels<DK, R>(g, kh, a.Hk, buf, c0, dst);
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
        setup_barrier(32 * SW);
        if (warp == 1 && !__any_sync(0xffffffffu, failed)) {
          GateRaw gr{};
          if (lane < R) {
            const int h = kh * R + lane;
            gr = gate_load(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                           static_cast<int64_t>(b) * a.Hv + h, h);
          }
          finish_setup<DK, R>(a, buf, gr, lane);
        }
        mbar_arrive(sfull0 + 8 * p);  // every setup thread: its writes are released
        ++n;
      }
    } else {
      // Each warp prepares whole units: active unit n goes to warp n % SW and
      // buffer n % NB. The loads of up to two conv groups per lane are in flight
      // before the warp waits for its buffer.
      constexpr int NGL = (NG + 31) / 32;  // conv groups per lane
      const int w = warp - 1;
      UnitSlots slots;
      for (int i = 0, u = blockIdx.x; u < num_units; ++i, u += G) {
        const int b = u / a.Hk, kh = u % a.Hk;
        const int32_t s = slots.get(a, i, num_units, lane);
        if (!unit_active(s, a.num_slots)) {
          if (s >= a.num_slots && w == 0 && lane == 0 && kh == 0 && a.err)
            atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
          continue;
        }
        const uint32_t my = n++;
        if (static_cast<int>(my % SW) != w) continue;
        const uint32_t p = my % NB, use = my / NB;
        float* buf = setup + p * Cfg::kSetupStride;
        GateRaw gr{};
        if (lane < R) {
          const int h = kh * R + lane;
          gr = gate_load(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                         static_cast<int64_t>(b) * a.Hv + h, h);
        }
        const uint16_t* xrow = static_cast<const uint16_t*>(a.mixed) + static_cast<int64_t>(b) * a.D;
        bool waited = false, failed = false;
#pragma unroll
        for (int j0 = 0; j0 < NGL; j0 += 2) {
          GroupLoads<kF32Cache> L[2];
          int c0[2];
          float* dst[2];
          bool on[2];
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int g = lane + 32 * (j0 + jj);
            on[jj] = (j0 + jj < NGL) && g < NG;
            c0[jj] = 0;
            dst[jj] = buf;
            if (on[jj]) {
              group_channels<DK, R>(g, kh, a.Hk, buf, c0[jj], dst[jj]);
              group_load<kF32Cache>(a, xrow, s, c0[jj], L[jj]);
            }
          }
          if (!waited) {  // the buffer must be free before it is written
            waited = true;
            if (!mbar_wait_bounded(sempty0 + 8 * p, (use & 1) ^ 1)) { failed = true; break; }
          }
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
            if (on[jj]) group_conv<kF32Cache>(a, s, c0[jj], L[jj], dst[jj]);
        }
        if (__any_sync(0xffffffffu, failed)) {  // the consumers time out on this buffer too
          if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
          return;
        }
        __syncwarp();
        finish_setup<DK, R>(a, buf, gr, lane);
        mbar_arrive(sfull0 + 8 * p);  // every lane: its writes are released
      }
    }
    return;
  }

  if (warp == Cfg::kEpiWarp) {
    // ------------------------------------------------------------ epilogue
    // Output gate (gated calls only): per active unit, wait for the consumers'
    // fp32 o in o buffer n % 2, then per value head
    //   out = o / sqrt(mean(o^2) + eps) * (w + offset) * act(z).
    // A lane takes 8-element chunks c = lane + 32 j of the unit's R*dv outputs;
    // the dv/8 lanes of one head sum o^2 with xor shuffles.
    if (!a.gated) return;
    constexpr int NCH = Cfg::kUnitRows / 8;
    constexpr int NCL = (NCH + 31) / 32;
    constexpr int LPH = DV / 8;  // lanes per head within one pass
    float wv[NCL][8];
#pragma unroll
    for (int j = 0; j < NCL; ++j) {
      const int c = lane + 32 * j;
      const int i0 = (8 * c) % DV;
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.gate_w + i0));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.gate_w + i0 + 4));
      const float wr[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) wv[j][e] = wr[e] + a.gate_offset;
    }
    UnitSlots slots;
    uint32_t n = 0;
    for (int i = 0, u = blockIdx.x; u < num_units; ++i, u += G) {
      const int b = u / a.Hk, kh = u % a.Hk;
      const int32_t s = slots.get(a, i, num_units, lane);
      if (!unit_active(s, a.num_slots)) continue;
      const uint32_t po = n & 1, use = n >> 1;
      const int64_t base = (static_cast<int64_t>(b) * a.Hv + kh * R) * DV;
      uint4 zr[NCL];
#pragma unroll
      for (int j = 0; j < NCL; ++j) {
        const int c = lane + 32 * j;
        zr[j] = c < NCH ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.gate_z) +
                                                               base + 8 * c))
                        : make_uint4(0u, 0u, 0u, 0u);
      }
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(ofull0 + 8 * po, use & 1))) {
        if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
        return;
      }
      const float* ob = obuf + po * Cfg::kUnitRows;
#pragma unroll
      for (int j = 0; j < NCL; ++j) {
        const int c = lane + 32 * j;
        const bool on = c < NCH;
        float ov[8];
        if (on) {
          const float4 o0 = reinterpret_cast<const float4*>(ob + 8 * c)[0];
          const float4 o1 = reinterpret_cast<const float4*>(ob + 8 * c)[1];
          ov[0] = o0.x; ov[1] = o0.y; ov[2] = o0.z; ov[3] = o0.w;
          ov[4] = o1.x; ov[5] = o1.y; ov[6] = o1.z; ov[7] = o1.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) ov[e] = 0.0f;
        }
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(ov[e], ov[e], ss);
#pragma unroll
        for (int m = LPH / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float den = __fadd_rn(__fdiv_rn(ss, static_cast<float>(DV)), a.gate_eps);
        const float inv = den > 0.0f ? 1.0f / sqrtf(den) : 0.0f;  // all-zero head, eps 0
        float z8[8], y[8];
        unpack8(zr[j], z8);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float act = a.gate_act == GDN_ACT_SIGMOID
                                ? __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z8[e])))
                                : silu_f(z8[e]);
          y[e] = ((ov[e] * inv) * wv[j][e]) * act;
        }
        if (on) {
          if (a.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + base + 8 * c);
            dst[0] = make_float4(y[0], y[1], y[2], y[3]);
            dst[1] = make_float4(y[4], y[5], y[6], y[7]);
          } else {
            uint4 pk;
            pk.x = pack_bf2(y[0], y[1]);
            pk.y = pack_bf2(y[2], y[3]);
            pk.z = pack_bf2(y[4], y[5]);
            pk.w = pack_bf2(y[6], y[7]);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + base + 8 * c) = pk;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(oempty0 + 8 * po);  // the consumers may refill this buffer
      ++n;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1 - SW;
  if (g_test_fault == 1 && blockIdx.x == 0 && cw == 0 &&
      !__all_sync(0xffffffffu, mbar_wait_bounded(dead, 0, kTestWaitNs))) {
    if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
    return;
  }
  constexpr int RPW = Cfg::kRowsPerWarp;
  uint32_t g = 0, n = 0;
  UnitSlots slots;
  for (int i = 0, u = blockIdx.x; u < num_units; ++i, u += G) {
    const int b = u / a.Hk, kh = u % a.Hk;
    const int32_t s = slots.get(a, i, num_units, lane);
    const int64_t out_base = (static_cast<int64_t>(b) * a.Hv + kh * R) * DV;
    if (!unit_active(s, a.num_slots)) {  // inactive / invalid row: zero outputs, no state touched
      for (int i = cw * 32 + lane; i < per_unit_rows; i += kConsumerWarps * 32) {
        if (a.out_f32) static_cast<float*>(a.out)[out_base + i] = 0.0f;
        else static_cast<uint16_t*>(a.out)[out_base + i] = 0;
      }
      continue;
    }
    const uint32_t p = n % NB;
    // warp-uniform waits: a timed-out warp leaves as a whole (it shuffles below)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(sfull0 + 8 * p, (n / NB) & 1))) {
      if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
      return;
    }
    const uint32_t po = n & 1;  // o buffer of a gated call
    if (a.gated &&
        !__all_sync(0xffffffffu, mbar_wait_bounded(oempty0 + 8 * po, ((n >> 1) & 1) ^ 1))) {
      if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
      return;
    }
    float* ob = obuf + po * Cfg::kUnitRows;
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
    unsigned char* dst_base = reinterpret_cast<unsigned char*>(a.ssm) +
                              (static_cast<int64_t>(s) * a.Hv + kh * R) * (DV * Cfg::kRowBytes);
    for (int k = 0; k < Cfg::kStagesPerUnit; ++k, ++g) {
      const uint32_t r = g % NS, c = g / NS;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * r, c & 1))) {
        if (lane == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
        return;
      }
      const int row0 = k * Cfg::kStageRows + cw * RPW;
      const int hl = row0 / DV;
      const float al = gb[hl], be = gb[R + hl];
      const unsigned char* src = ring + static_cast<size_t>(r) * Cfg::kStageBytes +
                                 cw * RPW * Cfg::kRowBytes;
      // this warp's rows -> registers; the stage goes back to the producer at once
      float sv[RPW][VPL];
#pragma unroll
      for (int i = 0; i < RPW; ++i) IO::load(src + i * Cfg::kRowBytes, lane, sv[i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * r);
      float delta, ov;
      int ri;
      bool writer;
      rows_predict<VPL, RPW>(sv, qv, kv, vb, row0, al, be, kq, lane, delta, ov, ri, writer);
      if (writer) {
        if (a.gated) ob[row0 + ri] = ov;  // the epilogue warp gates and stores it
        else if (a.out_f32) static_cast<float*>(a.out)[out_base + row0 + ri] = ov;
        else static_cast<uint16_t*>(a.out)[out_base + row0 + ri] = f2bf(ov);
      }
      rows_update_store<VPL, RPW, kBf16State>(
          sv, kv, al, delta, dst_base + static_cast<int64_t>(row0) * Cfg::kRowBytes,
          Cfg::kRowBytes, lane);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(sempty0 + 8 * p);  // this warp no longer reads the setup buffer
      if (a.gated) mbar_arrive(ofull0 + 8 * po);  // its o values are in the o buffer
    }
    ++n;
  }
}


// ------------------------------------------------------------------ small batches
// With fewer units than SMs the persistent kernel leaves most SMs idle and each busy one
// streams a whole unit. Here a unit (row b, k-head kh) is split over the P CTAs of a
// thread-block cluster instead: CTA p takes the unit's rows [p NR, (p + 1) NR), NR = R dv / P,
// as many rows per warp as the persistent kernel's consumers take, loaded straight into
// registers before anything else. Every CTA runs the
// conv of the unit's q and k channels itself, from the old windows, and the conv of its own
// rows' v channels, whose windows it rolls. CTA 0 rolls the q and k windows, after a
// cluster barrier that every CTA of the cluster arrives at once its window reads are done.
// The arithmetic of a row is the persistent kernel's (conv8_step, finish_setup,
// rows_predict, lane_update), so its results do not depend on which kernel ran it.
template <int DK, int R, bool kBf16State, int P>
struct SplitCfg {
  using Cfg = DecodeCfg<DK, R, kBf16State>;
  static constexpr int RPW = Cfg::kRowsPerWarp;  // the persistent kernel's rows per warp
  static constexpr int NR = R * DK / P;          // rows per CTA
  static constexpr int kThreads = NR / RPW * 32;
};

template <int DK, int R, bool kF32Cache, bool kBf16State, int P>
__global__ void __launch_bounds__(SplitCfg<DK, R, kBf16State, P>::kThreads, 1)
    split_decode_kernel(LayerArgs a) {
  using SC = SplitCfg<DK, R, kBf16State, P>;
  using Cfg = typename SC::Cfg;
  constexpr int DV = DK, VPL = DK / 32, UR = R * DV, NR = SC::NR, RPW = SC::RPW;
  constexpr int NW = NR / RPW;
  constexpr int QG = DK / 8, VG = NR / 8, NG = 2 * QG + VG;
  static_assert(NR % RPW == 0 && NR % 8 == 0 && NW * 32 >= NG, "one conv group per thread");
  __shared__ __align__(16) float buf[Cfg::kSetupStride];  // the persistent kernel's layout
  __shared__ float qkwin[2 * QG][8][kConvW - 1];           // rolled q, k windows (CTA 0)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = blockIdx.x;  // the CTA's rank in its cluster (cluster = P x 1 x 1)
  const int u = blockIdx.y, b = u / a.Hk, kh = u % a.Hk;
  const int32_t s = a.slot[b];
  const int64_t out_base = (static_cast<int64_t>(b) * a.Hv + kh * R) * DV + part * NR;
  if (!unit_active(s, a.num_slots)) {  // the same for the whole cluster: no barrier is used
    if (s >= a.num_slots && part == 0 && kh == 0 && tid == 0 && a.err)
      atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
    for (int i = tid; i < NR; i += NW * 32) {
      if (a.out_f32) static_cast<float*>(a.out)[out_base + i] = 0.0f;
      else static_cast<uint16_t*>(a.out)[out_base + i] = 0;
    }
    return;
  }
  const int row0 = part * NR + warp * RPW;  // the warp's first row within the unit
  unsigned char* rows = reinterpret_cast<unsigned char*>(a.ssm) +
                        ((static_cast<int64_t>(s) * a.Hv + kh * R) * DV + row0) * Cfg::kRowBytes;
  float sv[RPW][VPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i)
    StateIO<VPL, kBf16State>::load(rows + i * Cfg::kRowBytes, lane, sv[i]);
  GateRaw gr{};
  if (warp == 0 && lane < R) {
    const int h = kh * R + lane;
    gr = gate_load(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias, static_cast<int64_t>(b) * a.Hv + h, h);
  }
  // one conv group per thread: q and k groups 0 .. 2 QG - 1, then this CTA's v groups
  if (tid < NG) {
    const bool qk = tid < 2 * QG;
    int c0;
    float* dst;
    if (qk) {
      group_channels<DK, R>(tid, kh, a.Hk, buf, c0, dst);
    } else {
      const int j = part * NR + 8 * (tid - 2 * QG);  // unit-relative v channel
      c0 = 2 * a.Hk * DK + kh * UR + j;
      dst = buf + 2 * DK + j;
    }
    float x8[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.mixed) +
                                                 static_cast<int64_t>(b) * a.D + c0)),
            x8);
    if (a.conv_w) {
      float win[8][kConvW - 1], y8[8];
      load_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, win);
      conv8_step<kF32Cache>(win, x8, static_cast<const uint16_t*>(a.conv_w),
                            static_cast<const uint16_t*>(a.conv_b), c0, a.silu != 0, y8);
      if (qk) {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
#pragma unroll
          for (int j = 0; j < kConvW - 1; ++j) qkwin[tid][ch][j] = win[ch][j];
      } else {
        store_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, win);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = y8[i];
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = x8[i];
    }
  }
  cluster_arrive();  // this CTA has read every window it needs
  __syncthreads();
  if (warp == 0) finish_setup<DK, R>(a, buf, gr, lane);
  __syncthreads();
  {
    float qv[VPL], kv[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
      qv[e] = buf[lane * VPL + e];
      kv[e] = buf[DK + lane * VPL + e];
    }
    const float* vb = buf + 2 * DK;
    const float* gb = buf + 2 * DK + UR;
    const int hl = row0 / DV;
    const float al = gb[hl], be = gb[R + hl], kq = gb[2 * R];
    float delta, ov;
    int ri;
    bool writer;
    rows_predict<VPL, RPW>(sv, qv, kv, vb, row0, al, be, kq, lane, delta, ov, ri, writer);
    if (writer) {
      const int64_t o = out_base + warp * RPW + ri;
      if (a.out_f32) static_cast<float*>(a.out)[o] = ov;
      else static_cast<uint16_t*>(a.out)[o] = f2bf(ov);
    }
    rows_update_store<VPL, RPW, kBf16State>(sv, kv, al, delta, rows, Cfg::kRowBytes, lane);
  }
  cluster_wait();  // every CTA of the cluster is past its window reads
  if (part == 0 && a.conv_w && tid < 2 * QG) {
    int c0;
    float* dst;
    group_channels<DK, R>(tid, kh, a.Hk, buf, c0, dst);
    float win[8][kConvW - 1];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
#pragma unroll
      for (int j = 0; j < kConvW - 1; ++j) win[ch][j] = qkwin[tid][ch][j];
    store_conv8<kF32Cache>(a.conv_state, a.conv_layout, s, a.D, c0, win);
  }
}

// CTAs per unit for a call: 1 runs the persistent kernel. Calls that fill the GPU, gated
// calls (the gate needs a whole head's o) and calls capped to part of the GPU (the mixed
// step) take the persistent kernel.
// Measured on GB300 (Qwen3-Next geometry, L2 flushed): the split kernel wins while a call
// has at most half as many units as SMs (B <= 4: 10.4-12.2 us against 12.7-13.7 us for the
// persistent kernel, fp32 state; ~10.3 against ~14 us with a bf16 state), P = 4 and P = 8
// within 0.3 us of each other; from B = 8 the persistent kernel, which overlaps its setup
// and streaming, is faster (14.6 against 17-18.5 us). Rows per CTA stay within [16, 128].
template <int DK, int R>
constexpr bool split_ok(int P) {
  return R * DK / P >= 16 && R * DK / P <= 128 && P <= 8;
}
template <int DK, int R>
int split_parts(const LayerArgs& a, int B) {
  if (a.gated || a.max_ctas > 0) return 1;
  const int64_t units = static_cast<int64_t>(B) * a.Hk;
  if (units * 2 > sm_count()) return 1;
  for (int p : {4, 8, 2})
    if (split_ok<DK, R>(p)) return p;
  return 1;
}

template <int DK, int R, bool kF32Cache, bool kBf16State, int P>
cudaError_t launch_split(const LayerArgs& a, int B, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P, static_cast<unsigned>(B) * a.Hk, 1);
  cfg.blockDim = dim3(SplitCfg<DK, R, kBf16State, P>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_decode_kernel<DK, R, kF32Cache, kBf16State, P>, a);
}

template <int DK, int R, bool kF32Cache, bool kBf16State>
cudaError_t launch_one(const LayerArgs& a, int B, cudaStream_t s) {
  using Cfg = DecodeCfg<DK, R, kBf16State>;
  switch (split_parts<DK, R>(a, B)) {
    case 2:
      if constexpr (split_ok<DK, R>(2)) return launch_split<DK, R, kF32Cache, kBf16State, 2>(a, B, s);
      break;
    case 4:
      if constexpr (split_ok<DK, R>(4)) return launch_split<DK, R, kF32Cache, kBf16State, 4>(a, B, s);
      break;
    case 8:
      if constexpr (split_ok<DK, R>(8)) return launch_split<DK, R, kF32Cache, kBf16State, 8>(a, B, s);
      break;
    default: break;
  }
  auto kern = decode_kernel<DK, R, kF32Cache, kBf16State>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int units = B * a.Hk;
  int grid = units < sm_count() ? units : sm_count();
  if (a.max_ctas > 0 && grid > a.max_ctas) grid = a.max_ctas;
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, s>>>(a, units);
  return cudaGetLastError();
}

template <int DK, int R>
cudaError_t launch_dk_r(const LayerArgs& a, int B, cudaStream_t s) {
  if (a.ssm_bf16) {
    if (a.conv_f32) return launch_one<DK, R, true, true>(a, B, s);
    return launch_one<DK, R, false, true>(a, B, s);
  }
  if (a.conv_f32) return launch_one<DK, R, true, false>(a, B, s);
  return launch_one<DK, R, false, false>(a, B, s);
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

cudaError_t set_decode_test_fault(int mode) {
  return cudaMemcpyToSymbol(g_test_fault, &mode, sizeof(int));
}

cudaError_t launch_decode(const LayerArgs& a, int B, cudaStream_t s) {
  switch (a.dk) {
    case 32: return launch_dk<32>(a, B, s);
    case 64: return launch_dk<64>(a, B, s);
    case 128: return launch_dk<128>(a, B, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
