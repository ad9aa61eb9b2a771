// gdn_prefill.cu -- chunked (UT/WY) prefill of the gated delta rule over
// packed variable-length sequences.
//
// Source: vLLM PR #53864 (CuteDSL GDN prefill), "Numerical root cause and
// fix": the prefill works on chunks, forms the lower-triangular per-chunk
// KK^T block and inverts it; three bf16 Newton-Schulz rounds were not enough
// on correlated keys. Here the unit lower-triangular system is SOLVED EXACTLY
// in fp32 by forward substitution (no iteration, no bf16 intermediate).
//
// Algebra (unrolling S_t = a_t S_{t-1} + b_t (v_t - a_t S_{t-1} k_t) k_t^T
// inside a chunk that starts from S0; G_t = running sum of g in the chunk):
//   A_tj = beta_t exp(G_t - G_j) (k_t . k_j), j < t
//   [U | W] = (I + A)^-1 [diag(beta) V | diag(beta exp(G)) K]
//   D = U - W S0^T
//   O = diag(exp(G)) Q S0^T + P D,  P_tj = exp(G_t - G_j) (q_t . k_j), j <= t
//   S_end = exp(G_last) S0 + D^T diag(exp(G_last - G_j)) K
// Every decay is an exp of a difference G_t - G_j <= 0, so nothing overflows
// and long decays underflow to zero as they should.
//
// Kernels:
//   prep   (1 CTA)            validate cu_seqlens, per-sequence slot check,
//                             chunk table (chunks are anchored at each
//                             sequence's start, so results do not depend on
//                             how sequences are packed)
//   conv   (gdn_conv.cu)      conv outputs to workspace, final conv windows
//   intra  (chunk, v-head)    norms, gates, KK^T, QK^T, the triangular solve;
//                             writes W, U, P, G to workspace -- fully parallel
//   pass   (seq, v-head, dv-slice)  sequential over the sequence's chunks:
//                             D, O and the state update with S in shared memory
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

namespace {

constexpr int kCMax = 64;
constexpr int kPreThreads = 256;
constexpr int kDvSplitMax = 4;

struct WsLayout {
  size_t meta, seq_ok, chunk_off, chunk_seq, ybuf, W, U, P, G, total;
  int max_chunks;
};

__host__ __device__ inline size_t align_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int T, int N, int Hv, int dk, int dv, int C, int conv, int D) {
  WsLayout L;
  const int64_t mc = (static_cast<int64_t>(T) + static_cast<int64_t>(N) * (C - 1)) / C;
  L.max_chunks = static_cast<int>(mc);
  size_t off = 0;
  L.meta = off; off = align_up(off + 16 * sizeof(int32_t));
  L.seq_ok = off; off = align_up(off + static_cast<size_t>(N) * sizeof(int32_t));
  L.chunk_off = off; off = align_up(off + static_cast<size_t>(N + 1) * sizeof(int32_t));
  L.chunk_seq = off; off = align_up(off + static_cast<size_t>(mc + 1) * sizeof(int32_t));
  L.ybuf = off; off = align_up(off + (conv ? static_cast<size_t>(T) * D * sizeof(uint16_t) : 0));
  // per-chunk tiles are stored with kCMax rows whatever the chunk size C
  const size_t ch = static_cast<size_t>(mc) * Hv * kCMax;
  L.W = off; off = align_up(off + ch * dk * sizeof(float));
  L.U = off; off = align_up(off + ch * dv * sizeof(float));
  L.P = off; off = align_up(off + ch * kCMax * sizeof(float));
  L.G = off; off = align_up(off + ch * sizeof(float));
  L.total = off;
  return L;
}

// ---------------------------------------------------------------- prep
constexpr int kOrderMaxSeqs = 1024;  // sequences ranked by length; identity order beyond
constexpr int kPrepThreads = 1024;

// Inclusive sum of v over the block (kPrepThreads threads), in a fixed order.
__device__ __forceinline__ int block_scan_incl(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int r = v + (warp > 0 ? s_warp[warp - 1] : 0);
  __syncthreads();  // s_warp free for the next call
  return r;
}

// The chunk table of a prefill call, one CTA. Every step is parallel over sequences or chunks
// and works in shared memory: the call's first kernels wait for it.
__global__ void __launch_bounds__(kPrepThreads)
    prep_kernel(LayerArgs a, PrefillExtra p, int32_t* meta, int32_t* seq_ok, int32_t* chunk_off,
                int32_t* chunk_seq, int32_t* seq_order) {
  __shared__ int s_bad;
  __shared__ int s_warp[32];
  __shared__ int s_off[kOrderMaxSeqs + 1];  // chunk_off, when N <= kOrderMaxSeqs
  const int N = p.num_seqs, C = p.chunk, tid = threadIdx.x;
  // a kernel launched as a programmatic dependent of this one may start now; it waits for this
  // grid's completion before it reads the tables
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // cu_seqlens: starts at 0, ends at total_tokens, never decreases
  for (int i = tid; i <= N; i += kPrepThreads) {
    const int v = p.cu_seqlens[i];
    const bool bad = (i == 0 && v != 0) || (i == N && v != p.total_tokens) ||
                     (i < N && p.cu_seqlens[i + 1] < v);
    if (bad) s_bad = 1;
  }
  __syncthreads();
  const bool valid = s_bad == 0;
  if (tid == 0 && !valid && a.err) atomicOr(a.err, GDN_DEVERR_SEQLENS);
  const bool small = N <= kOrderMaxSeqs;
  // per sequence: active or not, its chunk count; chunk_off by a running block scan
  int carry = 0;
  if (tid == 0) chunk_off[0] = 0;
  if (small && tid == 0) s_off[0] = 0;
  for (int b = 0; b < N; b += kPrepThreads) {
    const int i = b + tid;
    int cnt = 0;
    if (i < N) {
      const int32_t sl = a.slot[i];
      if (sl >= a.num_slots && a.err) atomicOr(a.err, GDN_DEVERR_SLOT_RANGE);
      const bool ok = valid && sl > 0 && sl < a.num_slots;
      seq_ok[i] = ok;
      if (ok) cnt = (p.cu_seqlens[i + 1] - p.cu_seqlens[i] + C - 1) / C;
    }
    const int incl = carry + block_scan_incl(cnt, s_warp);
    if (i < N) {
      chunk_off[i + 1] = incl;
      if (small) s_off[i + 1] = incl;
    }
    if (tid == kPrepThreads - 1) s_warp[0] = incl;  // the tile's last prefix: the next carry
    __syncthreads();
    carry = s_warp[0];
    __syncthreads();
  }
  if (tid == 0) meta[0] = carry;
  __syncthreads();  // chunk_off (global) and s_off visible to the block
  // chunk_seq[c]: the last sequence whose first chunk is at or before c
  const int32_t* off = small ? s_off : chunk_off;
  for (int c = tid; c < carry; c += kPrepThreads) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= c) lo = mid;
      else hi = mid - 1;
    }
    chunk_seq[c] = lo;
  }
  if (seq_order == nullptr) return;
  // seq_order[r] = the sequence of rank r by descending chunk count (ties by index): a state
  // pass launched in this order starts its longest chains first
  if (!small) {
    for (int i = tid; i < N; i += kPrepThreads) seq_order[i] = i;
    return;
  }
  for (int i = tid; i < N; i += kPrepThreads) {
    const int ci = s_off[i + 1] - s_off[i];
    int r = 0;
    for (int j = 0; j < N; ++j) {
      const int cj = s_off[j + 1] - s_off[j];
      r += (cj > ci) || (cj == ci && j < i);
    }
    seq_order[r] = i;
  }
}

// ---------------------------------------------------------------- intra-chunk
// One CTA per (chunk, v-head). Shared: q^, k^ [C][DK+1]; X = [beta V | beta e^G K]
// [C][DV+DK+1] solved in place; A [C][C+1]; G, beta [C].
template <int DK>
__global__ void __launch_bounds__(kPreThreads)
    intra_kernel(LayerArgs a, PrefillExtra p, const uint16_t* y, const int32_t* meta,
                 const int32_t* chunk_off, const int32_t* chunk_seq, float* Wb, float* Ub,
                 float* Pb, float* Gb) {
  constexpr int DV = DK;
  constexpr int KP = DK + 1, XP = DV + DK + 1, AP = kCMax + 1;
  extern __shared__ float sm[];
  float* Qh = sm;                 // [C][KP]
  float* Kh = Qh + kCMax * KP;    // [C][KP]
  float* X = Kh + kCMax * KP;     // [C][XP]
  float* A = X + kCMax * XP;      // [C][AP]
  float* Gs = A + kCMax * AP;     // [C]
  float* Bs = Gs + kCMax;         // [C]
  float* inv = Bs + kCMax;        // [2][C]

  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= meta[0]) return;
  const int C = p.chunk;
  const int i = chunk_seq[c];
  const int t0 = p.cu_seqlens[i] + (c - chunk_off[i]) * C;
  const int L = min(C, p.cu_seqlens[i + 1] - t0);
  const int kh = h / (a.Hv / a.Hk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qc = kh * DK, kc = (a.Hk + kh) * DK, vc = 2 * a.Hk * DK + h * DV;

  // load q, k, v (bf16) for L tokens; zero the tail rows
  for (int idx = tid; idx < kCMax * (DK / 8); idx += kPreThreads) {
    const int t = idx / (DK / 8), c8 = (idx % (DK / 8)) * 8;
    float qf[8], kf[8];
    if (t < L) {
      const uint16_t* row = y + static_cast<int64_t>(t0 + t) * a.D;
      unpack8(__ldg(reinterpret_cast<const uint4*>(row + qc + c8)), qf);
      unpack8(__ldg(reinterpret_cast<const uint4*>(row + kc + c8)), kf);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[e] = kf[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) { Qh[t * KP + c8 + e] = qf[e]; Kh[t * KP + c8 + e] = kf[e]; }
  }
  for (int idx = tid; idx < kCMax * (DV / 8); idx += kPreThreads) {
    const int t = idx / (DV / 8), c8 = (idx % (DV / 8)) * 8;
    float vf[8];
    if (t < L) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(y + static_cast<int64_t>(t0 + t) * a.D + vc + c8)), vf);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) vf[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) X[t * XP + c8 + e] = vf[e];
  }
  if (tid < kCMax) {
    float g = 0.0f, be = 0.0f;
    if (tid < L) gate_log(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                          static_cast<int64_t>(t0 + tid) * a.Hv + h, h, g, be);
    Gs[tid] = g;
    Bs[tid] = be;
  }
  __syncthreads();
  // norms: one warp per token row
  for (int t = warp; t < kCMax; t += kPreThreads / 32) {
    float sq = 0.0f, sk = 0.0f;
    for (int e = lane; e < DK; e += 32) {
      const float qx = Qh[t * KP + e], kx = Kh[t * KP + e];
      sq = fmaf(qx, qx, sq);
      sk = fmaf(kx, kx, sk);
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    if (lane == 0) {
      inv[t] = a.qk_l2norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
      inv[kCMax + t] = a.qk_l2norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
    }
  }
  if (tid == 0) {  // running sum of g (fixed order)
    float run = 0.0f;
    for (int t = 0; t < kCMax; ++t) { run += (t < L) ? Gs[t] : 0.0f; Gs[t] = run; }
  }
  __syncthreads();
  for (int idx = tid; idx < kCMax * DK; idx += kPreThreads) {
    const int t = idx / DK, e = idx % DK;
    Qh[t * KP + e] = (Qh[t * KP + e] * inv[t]) * a.scale;
    Kh[t * KP + e] = Kh[t * KP + e] * inv[kCMax + t];
  }
  __syncthreads();
  // RHS: X[:, 0:DV] = beta V ; X[:, DV:DV+DK] = beta e^G K
  for (int idx = tid; idx < kCMax * (DV + DK); idx += kPreThreads) {
    const int t = idx / (DV + DK), col = idx % (DV + DK);
    const float bt = Bs[t];
    if (col < DV) X[t * XP + col] = bt * X[t * XP + col];
    else X[t * XP + col] = (bt * expf(Gs[t])) * Kh[t * KP + (col - DV)];
  }
  // A (strictly lower) and P (lower incl. diagonal)
  float* Pout = Pb + (static_cast<int64_t>(c) * a.Hv + h) * kCMax * kCMax;
  for (int idx = tid; idx < kCMax * kCMax; idx += kPreThreads) {
    const int t = idx / kCMax, j = idx % kCMax;
    float kk = 0.0f, qk = 0.0f;
    if (j <= t && t < L) {
#pragma unroll 8
      for (int e = 0; e < DK; ++e) {
        const float kj = Kh[j * KP + e];
        kk = fmaf(Kh[t * KP + e], kj, kk);
        qk = fmaf(Qh[t * KP + e], kj, qk);
      }
    }
    const float dec = (j <= t && t < L) ? expf(Gs[t] - Gs[j]) : 0.0f;
    A[t * AP + j] = (j < t) ? Bs[t] * dec * kk : 0.0f;
    Pout[idx] = dec * qk;
  }
  __syncthreads();
  // forward substitution, one column of X per thread: X_r -= sum_{j<r} A_rj X_j
  for (int col = tid; col < DV + DK; col += kPreThreads) {
    for (int r = 1; r < L; ++r) {
      float s0 = 0.0f, s1 = 0.0f;
      int j = 0;
      for (; j + 1 < r; j += 2) {
        s0 = fmaf(A[r * AP + j], X[j * XP + col], s0);
        s1 = fmaf(A[r * AP + j + 1], X[(j + 1) * XP + col], s1);
      }
      if (j < r) s0 = fmaf(A[r * AP + j], X[j * XP + col], s0);
      X[r * XP + col] -= (s0 + s1);
    }
  }
  __syncthreads();
  float* Wout = Wb + (static_cast<int64_t>(c) * a.Hv + h) * kCMax * DK;
  float* Uout = Ub + (static_cast<int64_t>(c) * a.Hv + h) * kCMax * DV;
  for (int idx = tid; idx < kCMax * DV; idx += kPreThreads) {
    const int t = idx / DV, col = idx % DV;
    Uout[idx] = X[t * XP + col];
  }
  for (int idx = tid; idx < kCMax * DK; idx += kPreThreads) {
    const int t = idx / DK, col = idx % DK;
    Wout[idx] = X[t * XP + DV + col];
  }
  if (tid < kCMax) Gb[(static_cast<int64_t>(c) * a.Hv + h) * kCMax + tid] = Gs[tid];
}

// ---------------------------------------------------------------- state pass
// One CTA per (sequence, v-head, dv-slice of DVS rows). Shared: S [DVS][DK+1],
// W [C][DK+1], Qs = e^G q^ [C][DK+1], Ks = e^(G_last-G) k^ [C][DK+1],
// P [C][C+1], U/D [C][DVS+1].
template <int DK, int DVS>
__global__ void __launch_bounds__(kPreThreads)
    pass_kernel(LayerArgs a, PrefillExtra p, const uint16_t* y, const int32_t* seq_ok,
                const int32_t* chunk_off, const float* Wb, const float* Ub, const float* Pb,
                const float* Gb) {
  constexpr int DV = DK;
  constexpr int KP = DK + 1, PP = kCMax + 1, DP = DVS + 1;
  extern __shared__ float sm[];
  float* Ss = sm;                   // [DVS][KP]
  float* Ws = Ss + DVS * KP;        // [C][KP]
  float* Qs = Ws + kCMax * KP;      // [C][KP]
  float* Ks = Qs + kCMax * KP;      // [C][KP]
  float* Ps = Ks + kCMax * KP;      // [C][PP]
  float* Ds = Ps + kCMax * PP;      // [C][DP]
  float* Gs = Ds + kCMax * DP;      // [C]
  float* inv = Gs + kCMax;          // [2][C]

  const int i = blockIdx.x, h = blockIdx.y, sp = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bos = p.cu_seqlens[i], eos = p.cu_seqlens[i + 1];
  const int r0 = sp * DVS;
  if (!seq_ok[i]) {  // inactive / invalid sequence (or bad cu_seqlens): zero outputs
    int64_t n = static_cast<int64_t>(max(eos - bos, 0));
    if (bos < 0 || eos > p.total_tokens) n = 0;
    for (int64_t idx = tid; idx < n * DVS; idx += kPreThreads) {
      const int64_t t = bos + idx / DVS;
      const int64_t o = (t * a.Hv + h) * DV + r0 + idx % DVS;
      if (a.out_f32) static_cast<float*>(a.out)[o] = 0.0f;
      else static_cast<uint16_t*>(a.out)[o] = 0;
    }
    return;
  }
  const int C = p.chunk;
  const int kh = h / (a.Hv / a.Hk);
  const int32_t slot = a.slot[i];
  const bool init = (p.has_init == nullptr) || (p.has_init[i] != 0);
  const int64_t soff = (static_cast<int64_t>(slot) * a.Hv + h) * DV * DK + static_cast<int64_t>(r0) * DK;
  float* Sg = a.ssm + soff;                                  // fp32 state
  uint16_t* Sb = reinterpret_cast<uint16_t*>(a.ssm) + soff;  // bf16 state
  for (int idx = tid; idx < DVS * DK; idx += kPreThreads)
    Ss[(idx / DK) * KP + idx % DK] = init ? (a.ssm_bf16 ? bf2f(Sb[idx]) : Sg[idx]) : 0.0f;

  const int qc = kh * DK, kc = (a.Hk + kh) * DK;
  for (int c = chunk_off[i]; c < chunk_off[i + 1]; ++c) {
    const int t0 = bos + (c - chunk_off[i]) * C;
    const int L = min(C, eos - t0);
    const int64_t ch = static_cast<int64_t>(c) * a.Hv + h;
    __syncthreads();  // previous chunk's readers of the shared tiles are done
    for (int idx = tid; idx < kCMax * DK; idx += kPreThreads) {
      const int t = idx / DK, e = idx % DK;
      Ws[t * KP + e] = Wb[ch * kCMax * DK + idx];
    }
    for (int idx = tid; idx < kCMax * kCMax; idx += kPreThreads)
      Ps[(idx / kCMax) * PP + idx % kCMax] = Pb[ch * kCMax * kCMax + idx];
    for (int idx = tid; idx < kCMax * DVS; idx += kPreThreads) {
      const int t = idx / DVS, r = idx % DVS;
      Ds[t * DP + r] = Ub[ch * kCMax * DV + static_cast<int64_t>(t) * DV + r0 + r];
    }
    if (tid < kCMax) Gs[tid] = Gb[ch * kCMax + tid];
    for (int idx = tid; idx < kCMax * (DK / 8); idx += kPreThreads) {
      const int t = idx / (DK / 8), c8 = (idx % (DK / 8)) * 8;
      float qf[8], kf[8];
      if (t < L) {
        const uint16_t* row = y + static_cast<int64_t>(t0 + t) * a.D;
        unpack8(__ldg(reinterpret_cast<const uint4*>(row + qc + c8)), qf);
        unpack8(__ldg(reinterpret_cast<const uint4*>(row + kc + c8)), kf);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[e] = kf[e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) { Qs[t * KP + c8 + e] = qf[e]; Ks[t * KP + c8 + e] = kf[e]; }
    }
    __syncthreads();
    for (int t = warp; t < kCMax; t += kPreThreads / 32) {
      float sq = 0.0f, sk = 0.0f;
      for (int e = lane; e < DK; e += 32) {
        const float qx = Qs[t * KP + e], kx = Ks[t * KP + e];
        sq = fmaf(qx, qx, sq);
        sk = fmaf(kx, kx, sk);
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      if (lane == 0) {
        inv[t] = a.qk_l2norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
        inv[kCMax + t] = a.qk_l2norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
      }
    }
    __syncthreads();
    const float Glast = Gs[L - 1];
    for (int idx = tid; idx < kCMax * DK; idx += kPreThreads) {
      const int t = idx / DK, e = idx % DK;
      const bool live = t < L;
      Qs[t * KP + e] = live ? ((Qs[t * KP + e] * inv[t]) * a.scale) * expf(Gs[t]) : 0.0f;
      Ks[t * KP + e] = live ? (Ks[t * KP + e] * inv[kCMax + t]) * expf(Glast - Gs[t]) : 0.0f;
    }
    __syncthreads();
    // D = U - W S^T   (thread: r = lane (< DVS), rows t = warp + 8 m)
    float o_acc[kCMax / (kPreThreads / 32)];
    {
      constexpr int TPW = kCMax / (kPreThreads / 32);
      const int r = lane % DVS;
      const bool act = lane < DVS;
      float dacc[TPW];
#pragma unroll
      for (int m = 0; m < TPW; ++m) { dacc[m] = 0.0f; o_acc[m] = 0.0f; }
      if (act) {
        for (int e = 0; e < DK; ++e) {
          const float sre = Ss[r * KP + e];
#pragma unroll
          for (int m = 0; m < TPW; ++m) {
            const int t = warp + 8 * m;
            dacc[m] = fmaf(Ws[t * KP + e], sre, dacc[m]);
            o_acc[m] = fmaf(Qs[t * KP + e], sre, o_acc[m]);
          }
        }
      }
      __syncthreads();
      if (act) {
#pragma unroll
        for (int m = 0; m < TPW; ++m) {
          const int t = warp + 8 * m;
          Ds[t * DP + r] = (t < L) ? Ds[t * DP + r] - dacc[m] : 0.0f;
        }
      }
      __syncthreads();
      // O = e^G Q S^T + P D, written out
      if (act) {
#pragma unroll
        for (int m = 0; m < TPW; ++m) {
          const int t = warp + 8 * m;
          float acc = o_acc[m];
          for (int j = 0; j <= t; ++j) acc = fmaf(Ps[t * PP + j], Ds[j * DP + r], acc);
          if (t < L) {
            const int64_t o = (static_cast<int64_t>(t0 + t) * a.Hv + h) * DV + r0 + r;
            if (a.out_f32) static_cast<float*>(a.out)[o] = acc;
            else static_cast<uint16_t*>(a.out)[o] = f2bf(acc);
          }
        }
      }
    }
    // S = e^G_last S + D^T Ks  (thread: column e = tid % DK, rows r = tid / DK + step)
    {
      const float gl = expf(Glast);
      constexpr int RSTEP = kPreThreads / DK > 0 ? kPreThreads / DK : 1;
      for (int idx = tid; idx < DVS * DK; idx += kPreThreads) {
        const int r = idx / DK, e = idx % DK;
        float acc = gl * Ss[r * KP + e];
        for (int t = 0; t < L; ++t) acc = fmaf(Ds[t * DP + r], Ks[t * KP + e], acc);
        Ss[r * KP + e] = acc;
      }
      (void)RSTEP;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < DVS * DK; idx += kPreThreads) {
    const float v = Ss[(idx / DK) * KP + idx % DK];
    if (a.ssm_bf16) Sb[idx] = f2bf(v);  // rounded to bf16 only here, at the write-back
    else Sg[idx] = v;
  }
}

template <int DK>
size_t intra_smem() {
  return sizeof(float) * (2 * kCMax * (DK + 1) + kCMax * (2 * DK + 1) + kCMax * (kCMax + 1) + 4 * kCMax);
}
template <int DK, int DVS>
size_t pass_smem() {
  return sizeof(float) * (DVS * (DK + 1) + 3 * kCMax * (DK + 1) + kCMax * (kCMax + 1) +
                          kCMax * (DVS + 1) + 3 * kCMax);
}

template <int DK>
cudaError_t launch_prefill_dk(const LayerArgs& a, const PrefillExtra& p, cudaStream_t s) {
  const WsLayout L = ws_layout(p.total_tokens, p.num_seqs, a.Hv, a.dk, a.dv, p.chunk,
                               a.conv_w != nullptr, a.D);
  char* ws = static_cast<char*>(p.workspace);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + L.meta);
  int32_t* seq_ok = reinterpret_cast<int32_t*>(ws + L.seq_ok);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_off);
  int32_t* chunk_seq = reinterpret_cast<int32_t*>(ws + L.chunk_seq);
  uint16_t* ybuf = reinterpret_cast<uint16_t*>(ws + L.ybuf);
  float* Wb = reinterpret_cast<float*>(ws + L.W);
  float* Ub = reinterpret_cast<float*>(ws + L.U);
  float* Pb = reinterpret_cast<float*>(ws + L.P);
  float* Gb = reinterpret_cast<float*>(ws + L.G);

  prep_kernel<<<1, kPrepThreads, 0, s>>>(a, p, meta, seq_ok, chunk_off, chunk_seq, nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const uint16_t* y = static_cast<const uint16_t*>(a.mixed);
  if (a.conv_w) {
    e = launch_prefill_conv(a, p, meta, seq_ok, chunk_off, chunk_seq, L.max_chunks, ybuf, s);
    if (e != cudaSuccess) return e;
    y = ybuf;
  }
  if (L.max_chunks > 0) {
    const size_t sm1 = intra_smem<DK>();
    cudaFuncSetAttribute(intra_kernel<DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm1));
    intra_kernel<DK><<<dim3(L.max_chunks, a.Hv), kPreThreads, sm1, s>>>(a, p, y, meta, chunk_off,
                                                                         chunk_seq, Wb, Ub, Pb, Gb);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  constexpr int DVS = DK / kDvSplitMax < 32 ? 32 : DK / kDvSplitMax;
  const size_t sm2 = pass_smem<DK, DVS>();
  cudaFuncSetAttribute(pass_kernel<DK, DVS>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm2));
  if (p.before_pass && (e = cudaEventRecord(p.before_pass, s)) != cudaSuccess) return e;
  if (p.num_seqs > 0)
    pass_kernel<DK, DVS><<<dim3(p.num_seqs, a.Hv, DK / DVS), kPreThreads, sm2, s>>>(
        a, p, y, seq_ok, chunk_off, Wb, Ub, Pb, Gb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_prep(const LayerArgs& a, const PrefillExtra& p, int32_t* meta,
                                int32_t* seq_ok, int32_t* chunk_off, int32_t* chunk_seq,
                                int32_t* seq_order, cudaStream_t s) {
  prep_kernel<<<1, kPrepThreads, 0, s>>>(a, p, meta, seq_ok, chunk_off, chunk_seq, seq_order);
  return cudaGetLastError();
}

size_t prefill_workspace_bytes(int total_tokens, int num_seqs, int Hk, int Hv, int dk, int dv,
                               int chunk, int conv) {
  if (dk == 128 && dv == 128) return prefill_tc_workspace_bytes(total_tokens, num_seqs, Hk, Hv, chunk);
  const int D = 2 * Hk * dk + Hv * dv;
  return ws_layout(total_tokens, num_seqs, Hv, dk, dv, chunk, conv, D).total;
}

cudaError_t launch_prefill(const LayerArgs& a, const PrefillExtra& p, cudaStream_t s) {
  cudaError_t e;
  switch (a.dk) {
    case 32: e = launch_prefill_dk<32>(a, p, s); break;
    case 64: e = launch_prefill_dk<64>(a, p, s); break;
    case 128: e = a.dv == 128 ? launch_prefill_tc(a, p, s) : launch_prefill_dk<128>(a, p, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || !a.gated) return e;
  // the output gate over every (token, value head) row of out, after the state pass
  return launch_output_gate(a, static_cast<int64_t>(p.total_tokens) * a.Hv, s);
}

}  // namespace gdn
