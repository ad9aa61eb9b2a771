// gdn_prefill_tc.cu -- chunked (UT/WY) prefill of the gated delta rule on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory), for
// dk = dv = 128 (the Qwen3-Next head size).
//
// Source: vLLM PR #53864 (CuteDSL GDN prefill), "Numerical root cause and
// fix": the prefill forms the per-chunk KK^T block and inverts the unit
// lower-triangular matrix built from it; a bf16 Newton-Schulz inverse fails on
// correlated keys. Here that inverse is solved EXACTLY in fp32 (a blocked
// recursive inverse: 8 x 8 diagonal blocks by forward substitution, then blocks
// of 16, 32 and 64 rows as T21 = -T22 (A21 T11)), and every contraction runs on
// the tensor cores with fp32 accumulation.
//
// Algebra per chunk of C tokens starting from state S0 (G_t = running sum of g
// inside the chunk, raw bf16 q, k, v, inverse norms iq_t, ik_t):
//   A_tj = beta_t e^(G_t - G_j) ik_t ik_j (k_t . k_j),  j < t;  T = (I + A)^-1
//   U = T diag(beta) V                    W = T diag(beta e^G ik) K
//   P_tj = e^(G_t - G_j) iq_t scale ik_j (q_t . k_j),  j <= t
//   D = U - W S0^T,   O = diag(e^G iq scale) Q S0^T + P D
//   S_end = e^(G_last) S0 + D^T diag(e^(G_last - G_j) ik_j) K
// (the same identity as the CUDA-core path; unrolling the rule inside a chunk).
//
// Precision: raw q, k, v are bf16 and enter the tensor cores exactly. Every
// fp32 operand (T diag(beta), the state S, W, P, D) is split into bf16 hi + lo
// (x = hi + lo to ~2^-17) and a product of two split operands takes three MMAs
// (hi*hi + hi*lo + lo*hi), one split and one exact operand two. The error per
// product is ~1e-5 relative, well inside the prefill bound.
//
// Kernels (after the shared chunk table and conv):
//   intra (64 token rows = 64/C chunks of one k-head per CTA, two CTAs per SM):
//       one MMA over the stacked [K; Q] operand (M = 128, N = 64) gives KK^T
//       and QK^T of the 64 rows at once (the diagonal CxC blocks are the
//       chunks'), then per value head: gates, A and P rows from tensor memory,
//       the fp32 triangular solve, U and W as MMAs with a block-diagonal T.
//       Writes the pass's operand tiles, already in tensor-core layout, to
//       workspace.
//   pass (sequence, value head): the state S lives in registers (a thread owns
//       half a row), its bf16 hi / lo parts in tensor memory; per chunk, bulk
//       copies bring the chunk's tiles into shared memory, MMA group 1 forms
//       S W^T and S Q^T (the compute warps then form D^T = U^T - S W^T), MMA
//       group 2 the state update D'^T K and then O2 = D^T P^T onto f_t O1;
//       M = dv = 128 throughout. With few sequences the chunks run in pieces,
//       each piece's pass beside the next piece's intra kernel.
// Every wait is bounded (GDN_DEVERR_TIMEOUT on expiry, the CTA stops cleanly
// and frees its tensor memory).
#include <climits>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int kD = 128;          // dk = dv

// Programmatic dependent launch. grid_dep_launch: once every CTA of this grid has executed it
// (or exited), the next kernel of the stream, if launched as a programmatic dependent, may
// start. grid_dep_wait: waits until the grid this one was launched as a dependent of has
// completed and its memory is visible.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
constexpr int kThreadsTc = 256;  // 8 warps: warp w reads tensor-memory lanes 32 (w % 4) ..
// the pass kernel adds two warps: warp 8 (lane 0) issues the MMA groups, warp 9 (lane 0) the
// bulk copies. The copy warp paces itself on mbarriers alone; the other nine warps meet at
// a named barrier of kSyncThreads
constexpr int kPassThreads = kThreadsTc + 64;
constexpr int kSyncThreads = kThreadsTc + 32;
constexpr uint32_t kTmemCols = 512;

// Test hook (gdn_testing_set_fault, mode 2): compute warp 0 of the state pass's first CTA
// waits, with a 10 ms bound, on a barrier nothing arrives on in place of its first group-2
// wait, and reports it as a wait that ran out, so the pass's failure path runs on the GPU:
// the other warps leave the chunk loop while the next chunk's tiles may still be in flight.
__device__ int g_test_fault = 0;
constexpr uint64_t kTestWaitNs = 10000000ull;
constexpr int kVecFloats = 256;  // per (chunk, head): f[C], dd[C], g_last

// A prefill of at most kPieceSeqHeads (sequence, value head) pairs leaves most SMs free during
// its state pass; its chunks then run in pieces (launch_tc_c), the pass of one piece beside the
// intra kernel of the next, and a sequence's fp32 state crosses a piece boundary in `sx`.
constexpr int kPieceSeqHeads = 64;

struct TcLayout {
  size_t meta, seq_ok, chunk_off, chunk_seq, seq_order, ybuf, Qt, Kt, Wt, Pt, Ut, vec, sx, total;
  int max_chunks;
  // per-tile byte sizes
  size_t q_tile, w_tile, p_tile, u_tile;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

TcLayout tc_layout(int T, int N, int Hk, int Hv, int C, int D) {
  TcLayout L;
  const int64_t mc = (static_cast<int64_t>(T) + static_cast<int64_t>(N) * (C - 1)) / C;
  L.max_chunks = static_cast<int>(mc);
  L.q_tile = static_cast<size_t>(C) * kD * 2;  // bf16 [C x 128] (q and k tiles)
  L.w_tile = static_cast<size_t>(C) * kD * 2;  // one of hi / lo
  L.p_tile = static_cast<size_t>(C) * C * 2;   // one of hi / lo
  L.u_tile = static_cast<size_t>(kD) * C * 4;  // fp32 U^T [128 x C]
  size_t off = 0;
  L.meta = off; off = align256(off + 16 * sizeof(int32_t));
  L.seq_ok = off; off = align256(off + static_cast<size_t>(N) * sizeof(int32_t));
  L.chunk_off = off; off = align256(off + static_cast<size_t>(N + 1) * sizeof(int32_t));
  L.chunk_seq = off; off = align256(off + static_cast<size_t>(mc + 1) * sizeof(int32_t));
  L.seq_order = off; off = align256(off + static_cast<size_t>(N) * sizeof(int32_t));
  L.ybuf = off; off = align256(off + static_cast<size_t>(T) * D * sizeof(uint16_t));
  L.Qt = off; off = align256(off + static_cast<size_t>(mc) * Hk * L.q_tile);
  L.Kt = off; off = align256(off + static_cast<size_t>(mc) * Hk * L.q_tile);
  L.Wt = off; off = align256(off + static_cast<size_t>(mc) * Hv * 2 * L.w_tile);
  L.Pt = off; off = align256(off + static_cast<size_t>(mc) * Hv * 2 * L.p_tile);
  L.Ut = off; off = align256(off + static_cast<size_t>(mc) * Hv * L.u_tile);
  L.vec = off; off = align256(off + static_cast<size_t>(mc) * Hv * kVecFloats * 4);
  L.sx = off;
  if (static_cast<int64_t>(N) * Hv <= kPieceSeqHeads)
    off = align256(off + static_cast<size_t>(N) * Hv * kD * kD * 4);
  L.total = off;
  return L;
}

struct TcBufs {
  unsigned char* Qt;  // [chunk][Hk] bf16 q tile, K-major [C x 128]
  unsigned char* Kt;  // [chunk][Hk] bf16 k tile [C x 128], the q tile's layout (MN-major use)
  unsigned char* Wt;  // [chunk][Hv][hi, lo] bf16 W tile, K-major [C x 128]
  unsigned char* Pt;  // [chunk][Hv][hi, lo] bf16 P tile, K-major [C x C]
  float* Ut;          // [chunk][Hv] fp32 U^T [128 x C], laid out by u_image_offset
  float* vec;         // [chunk][Hv][256]: f[0..C), dd[64..64+C), g_last at [128]
  size_t q_tile, w_tile, p_tile;
};

// Byte offset of O(t, col) (token t, dv column col) in the pass kernel's bf16 output tile
// [C x 128]: the 16-byte pieces of a token row are XOR-swizzled by t & 7
__device__ __forceinline__ uint32_t out_tile_offset(int t, int col) {
  return static_cast<uint32_t>(t * 256 + (((col >> 3) ^ (t & 7)) << 4) + (col & 7) * 2);
}

// Byte offset of U^T(r, t) (state row r, token t of the chunk) in a U tile: the byte
// image of two bf16 [128 x C] K-major tiles, tokens t..t+3 of an 8-token group where the
// first tile holds (r, group), t+4..t+7 where the second does. The pass kernel's thread that
// owns row r reads a group as two 16-byte pieces, eight rows of a warp per 128 bytes, so
// its reads are free of bank conflicts.
__host__ __device__ __forceinline__ uint32_t u_image_offset(int r, int t, int C) {
  return static_cast<uint32_t>(((t >> 2) & 1) * (128 * C * 2)) + tc::kmajor_offset(r, t & ~7, C) +
         static_cast<uint32_t>((t & 3) * 4);
}

// fp32 -> bf16 hi + lo, 8 values (element i in bf16 slot i of each uint4): hi = bf16(x) and
// lo = bf16(x - hi), both round-to-nearest-even, so x ~= hi + lo to about 2^-17 relative.
// Pairs are converted at once.
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf2(x[2 * i], x[2 * i + 1]);
    const float r0 = x[2 * i] - __uint_as_float(h[i] << 16);
    const float r1 = x[2 * i + 1] - __uint_as_float(h[i] & 0xFFFF0000u);
    l[i] = pack_bf2(r0, r1);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

template <int N>
__device__ __forceinline__ void tmem_load(uint32_t addr, float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_load<8>(uint32_t addr, float (&v)[8]) { tc::tmem_ld8(addr, v); }
template <>
__device__ __forceinline__ void tmem_load<16>(uint32_t addr, float (&v)[16]) { tc::tmem_ld16(addr, v); }

// sync point between tensor-core work and threads: smem writes -> async proxy,
// tensor-memory reads done, CTA barrier. Returns true if any thread flagged `bad`.
__device__ __forceinline__ bool tc_sync(bool bad) {
  tc::fence_async_smem();
  tc::fence_before_sync();
  const int any = __syncthreads_or(bad ? 1 : 0);
  tc::fence_after_sync();
  return any != 0;
}

// tc_sync over the compute and MMA warps of the pass kernel (named barrier 1)
__device__ __forceinline__ bool pass_sync(bool bad) {
  tc::fence_async_smem();
  tc::fence_before_sync();
  uint32_t any;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, 1, %2, p;\n"
      "selp.u32 %0, 1, 0, q;\n}"
      : "=r"(any)
      : "r"(static_cast<uint32_t>(bad)), "n"(kSyncThreads)
      : "memory");
  tc::fence_after_sync();
  return any != 0;
}

// acc[i][j] += sum_k a[i][k] b[k][j] for RB x 4 fp32 blocks held as float4 rows (k = 0..3)
template <int RB>
__device__ __forceinline__ void fma_rows(float (&acc)[RB][4], const float4 (&a)[RB], const float4 (&b)[4]) {
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const float ai[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      acc[i][0] = fmaf(ai[kk], b[kk].x, acc[i][0]);
      acc[i][1] = fmaf(ai[kk], b[kk].y, acc[i][1]);
      acc[i][2] = fmaf(ai[kk], b[kk].z, acc[i][2]);
      acc[i][3] = fmaf(ai[kk], b[kk].w, acc[i][3]);
    }
  }
}

// Inclusive sum of v over the lanes of a chunk of C tokens within a warp (the whole warp for
// C >= 32; a C = 64 chunk's second warp then adds the first's total)
template <int C>
__device__ __forceinline__ float chunk_scan(float v, int lane) {
  constexpr int kSeg = C < 32 ? C : 32;
#pragma unroll
  for (int d = 1; d < kSeg; d <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, v, d);
    if ((lane & (kSeg - 1)) >= d) v += n;
  }
  return v;
}

// barrier of the intra kernel's four solver warps (warps 0-3; named barrier 1)
constexpr int kSolveThreads = 128;
__device__ __forceinline__ void solver_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// One level of the intra kernel's blocked inverse (the solver threads): every diagonal block of
// 2b rows of a chunk is built from its two b-row halves, already inverted in place, as
// T21 = -T22 (A21 T11), written over A21 (rows of stride SA floats, chunk-local columns). A
// thread takes RB rows x 4 columns of T21; the products skip the zero parts of the triangular
// factors (T11 has none above its diagonal, T22 none right of it).
template <int b, int C, int SA>
__device__ __forceinline__ void solve_merge(float* sA, int tid) {
  constexpr int RB = b == 32 ? 2 : 1;      // rows per thread
  constexpr int COLS = b / 4;              // 4-column groups of a row
  constexpr int PER = b * b / (4 * RB);    // threads per block
  constexpr int NT = (64 / (2 * b)) * PER;  // threads at work
  static_assert(NT <= kSolveThreads && NT % 32 == 0, "whole warps of the solver threads");
  const bool on = tid < NT;
  const int m = tid / PER, idx = tid % PER;
  const int R0 = 2 * b * m, o = R0 % C;
  const int j0 = 4 * (idx % COLS), i0 = RB * (idx / COLS);
  float* A21 = sA + (R0 + b + i0) * SA + o;  // the thread's row i: A21 + i SA
  float acc[RB][4];
#pragma unroll
  for (int i = 0; i < RB; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  if (on) {  // X = A21 T11: column block j0 needs rows l >= j0 of T11
    for (int l = j0; l < b; l += 4) {
      float4 av[RB], tv[4];
#pragma unroll
      for (int i = 0; i < RB; ++i) av[i] = *reinterpret_cast<const float4*>(A21 + i * SA + l);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tv[kk] = *reinterpret_cast<const float4*>(sA + (R0 + l + kk) * SA + o + j0);
      fma_rows<RB>(acc, av, tv);
    }
  }
  solver_sync();  // every A21 read: X takes its place
  if (on) {
#pragma unroll
    for (int i = 0; i < RB; ++i)
      *reinterpret_cast<float4*>(A21 + i * SA + j0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  solver_sync();
#pragma unroll
  for (int i = 0; i < RB; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  if (on) {  // T22 X: rows i0 .. i0 + RB - 1 of T22 need columns l < i0 + RB
    for (int l = 0; l < i0 + RB; l += 4) {
      float4 av[RB], xv[4];
#pragma unroll
      for (int i = 0; i < RB; ++i) av[i] = *reinterpret_cast<const float4*>(A21 + i * SA + b + l);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        xv[kk] = *reinterpret_cast<const float4*>(sA + (R0 + b + l + kk) * SA + o + j0);
      fma_rows<RB>(acc, av, xv);
    }
  }
  solver_sync();  // every X read: T21 takes its place
  if (on) {
#pragma unroll
    for (int i = 0; i < RB; ++i)
      *reinterpret_cast<float4*>(A21 + i * SA + j0) =
          make_float4(-acc[i][0], -acc[i][1], -acc[i][2], -acc[i][3]);
  }
}

// ============================================================== intra kernel
// A CTA takes 64 token rows (64 / C chunks) of one k-head, so that two CTAs fit on an SM
// (shared memory and 256 tensor-memory columns each) and each hides the other's latency.
// The raw products k_t . k_j and q_t . k_j do not depend on the value head, so one MMA over
// the stacked operand [K; Q] (M = 128) computes both once per CTA: tensor-memory lanes 0..63
// hold G = K K^T and lanes 64..127 QK = Q K^T, columns [0, 64). Per value head:
//   A rows (warps on lanes 0..63) and P rows (warps on lanes 64..127) from them,
//   the fp32 solve of T = (I + A)^-1 per chunk,
//   T' = T diag(beta) and T'' = T diag(beta e^G ik), both split into bf16 hi + lo,
//   U^T = V^T T'^T (columns [64, 128), a dv row per lane) with V raw bf16, and
//   W = T'' K (columns [128, 256), a token per lane) with K raw bf16 -- W = T diag(beta)
//   diag(e^G ik) K, the diagonal scaling moved onto T, so K enters exactly.
// The W MMA keeps M = 128: rows 64..127 of its A operand read the next buffer in shared
// memory, and those accumulator lanes are never read.
template <int C>
struct IntraSmem {
  static constexpr int kRows = 64;                   // token rows per CTA
  static constexpr int CPC = kRows / C;              // chunks per CTA
  static constexpr int kTile = kRows * 128 * 2;      // bf16 [64 x 128]
  static constexpr int kTT = kRows * kRows * 2;      // bf16 [64 x 64]
  // sK, sQ: raw k, q rows (K-major [64 x 128]), adjacent: together the [K; Q] operand;
  // sV: V rows (MN-major use, the same layout); sT2h/l: T'' (A operand of W), sT1h/l: T'
  // (B operand of U^T), K-major [64 x 64]. The W operands sT2h and sT2l are read 64 rows
  // past their ends, which must stay inside this block.
  static constexpr int oK = 0, oQ = kTile, oV = 2 * kTile;
  static constexpr int oT2h = 3 * kTile, oT2l = oT2h + kTT, oT1h = oT2l + kTT, oT1l = oT1h + kTT;
  // fp32 A [64][C + 4] (16-byte rows), then T in place; a row's 4 padding floats hold its
  // token's e^G ik, beta and q / k norm factors
  static constexpr int kSA = C + 4;
  static constexpr int oA = oT1l + kTT;
  static constexpr int oG = oA + kRows * kSA * 4;    // cumulative log-gates G: 64 floats
  static constexpr int oPart = oG + kRows * 4;       // partial squared norms [2][2][64]
  // per token: k's norm factor, the second value head's running gate sums (scanned within each
  // warp) and beta, computed during the first head's solve
  static constexpr int oTok = oPart + 4 * kRows * 4;
  static constexpr int oBar = oTok + 3 * kRows * 4, oTmem = oBar + 8, oT0 = oTmem + 8;
  static constexpr int kBytes = oT0 + 2 * CPC * 4;
  static_assert(oT1h - oT2h >= kTT && oT1l - oT2l >= kTT, "M = 128 reads stay in the block");
  static_assert(kBytes <= 113 * 1024, "two intra CTAs must fit on an SM");
};
constexpr uint32_t kIntraTmemCols = 256;
constexpr int kColGQ = 0, kColU = 64, kColW = 128;  // tensor-memory columns of G|QK, U^T, W

template <int C>
__global__ void __launch_bounds__(kThreadsTc, 2)
    intra_tc_kernel(LayerArgs a, PrefillExtra p, const uint16_t* __restrict__ y,
                    const int32_t* meta, const int32_t* chunk_off, const int32_t* chunk_seq,
                    TcBufs wb, int cta0, int chain, int hsplit, int pre_wait) {
  // cta0: the first CTA of this launch (a piece of the chunks). Every CTA, its work done, lets
  // the pass over the piece (a programmatic dependent of this grid) start its set-up. chain:
  // launched as a programmatic dependent of the pass over the piece before; CTA 0 then waits
  // for that pass before it exits, so that this grid -- which the pass over the piece waits
  // for -- completes only after it (the other CTAs leave at once and free their SM).
  // hsplit: the CTA takes the one value head blockIdx.z of its k-head (a launch that fits one
  // wave finishes in about half the time, each CTA repeating phase 1); otherwise all of them.
  // pre_wait: launched as a programmatic dependent of the kernel before it (the chunk table's,
  // or the conv's), whose results it waits for before reading anything.
  if (pre_wait) grid_dep_wait();
  using S = IntraSmem<C>;
  constexpr int CPC = S::CPC, NR = S::kRows;
  extern __shared__ __align__(1024) unsigned char sm[];
  float* sA = reinterpret_cast<float*>(sm + S::oA);
  constexpr int SA = S::kSA;
  float* s_G = reinterpret_cast<float*>(sm + S::oG);
  float* s_part = reinterpret_cast<float*>(sm + S::oPart);
  // after phase 1 the partial norms are consumed: the head loop keeps each token's beta and
  // beta e^G ik there, 16-byte rows for the T' / T'' scaling
  float* s_beta = s_part;
  float* s_bsc = s_part + NR;
  float* s_ik = reinterpret_cast<float*>(sm + S::oTok);
  float* s_G1 = s_ik + NR;
  float* s_beta1 = s_ik + 2 * NR;
  // per-token values in A's row padding
  constexpr int kBeta = 1, kIq = 2, kIk = 3;
  auto pad = [&](int t, int k) -> float& { return sA[t * SA + C + k]; };
  int* s_t0 = reinterpret_cast<int*>(sm + S::oT0);
  int* s_L = s_t0 + CPC;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + S::oTmem);
  const uint32_t bar = smem_addr(sm + S::oBar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kh = blockIdx.y;
  const int nchunks = meta[0];
  const int c_first = (cta0 + blockIdx.x) * CPC;
  const bool waits = chain && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  const int R = a.Hv / a.Hk;
  const int hr0 = hsplit ? static_cast<int>(blockIdx.z) : 0, hr1 = hsplit ? hr0 + 1 : R;
  if (c_first >= nchunks) {  // no chunk of this CTA exists
    grid_dep_launch();
    if (waits) grid_dep_wait();
    return;
  }
  if (tid < CPC) {
    const int c = c_first + tid;
    int t0 = 0, L = 0;
    if (c < nchunks) {
      const int i = chunk_seq[c];
      t0 = p.cu_seqlens[i] + (c - chunk_off[i]) * C;
      L = min(C, p.cu_seqlens[i + 1] - t0);
    }
    s_t0[tid] = t0;
    s_L[tid] = L;
  }
  __syncthreads();
  // the first value head's gate inputs of this thread's token row, loaded before phase 1 so
  // that their latency overlaps it
  GateRaw gr0{};
  if (tid < NR) {
    const int ci = tid / C, tl = tid % C, h0 = kh * R + hr0;
    if (tl < s_L[ci])
      gr0 = gate_load(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                      static_cast<int64_t>(s_t0[ci] + tl) * a.Hv + h0, h0);
  }

  // ---- phase 1: raw q, k rows -> tensor-core tiles; norms. Thread: token row tok, q or k,
  // half of the 128 channels ----
  {
    const int tok = tid & 63, which = (tid >> 6) & 1, hf = tid >> 7;
    const int ci = tok / C, tl = tok % C;
    const bool valid = tl < s_L[ci];
    const int col0 = (which ? (a.Hk + kh) * kD : kh * kD) + 64 * hf;
    unsigned char* tile = sm + (which ? S::oK : S::oQ);
    const uint16_t* row = y + static_cast<int64_t>(s_t0[ci] + tl) * a.D + col0;
    uint4 v[8];
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8)
      v[k8] = valid ? __ldg(reinterpret_cast<const uint4*>(row) + k8) : make_uint4(0u, 0u, 0u, 0u);
    float ss = 0.0f;
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) {
      float f[8];
      unpack8(v[k8], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
      *reinterpret_cast<uint4*>(tile + tc::kmajor_offset(tok, 64 * hf + 8 * k8, kD)) = v[k8];
    }
    s_part[(hf * 2 + which) * NR + tok] = ss;
  }
  if (CPC > 1) {  // block-diagonal T' and T'': the off-diagonal blocks stay zero
    for (int i = tid; i < 4 * S::kTT / 16; i += kThreadsTc)
      reinterpret_cast<uint4*>(sm + S::oT2h)[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == 0) {
    tc::tmem_alloc(s_tmem, kIntraTmemCols);
    // gives up this CTA's right to allocate again: until a CTA that may still allocate tensor
    // memory has done so, the SM starts no other such CTA (measured: one CTA per SM without
    // this, two with it)
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  tc_sync(false);
  const uint32_t tb = *s_tmem;
  if (tid == 0) {  // [K; Q] K^T: G in lanes 0..63, QK in lanes 64..127, once per CTA
    const uint32_t id = tc::idesc_bf16_f32(128, NR);
    const uint32_t ak = smem_addr(sm + S::oK);
    for (int ks = 0; ks < kD / 16; ++ks)
      tc::mma_bf16(tb + kColGQ, tc::kmajor_desc(ak, kD, ks), tc::kmajor_desc(ak, kD, ks), id, ks > 0);
    tc::mma_commit(bar);
  }
  if (tid < 2 * NR) {  // the two halves' sums, in a fixed order
    const int tok = tid & 63, which = tid >> 6;
    const float ss = s_part[which * NR + tok] + s_part[(2 + which) * NR + tok];
    const float inv = a.qk_l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    pad(tok, which ? kIk : kIq) = inv;
    if (which) s_ik[tok] = inv;
  }
  uint32_t phase = 0;
  bool bad = false;

  for (int hr = hr0; hr < hr1 && !bad; ++hr) {
    const int h = kh * R + hr;
    // gates of the 64 token rows (warps 0 and 1, a row per thread), then the running sums per
    // chunk: an inclusive scan over the lanes of a chunk (C <= 32: inside a warp; C = 64: each
    // warp, then the second adds the first's total)
    if (tid < NR) {
      const int ci = tid / C, tl = tid % C;
      float g = 0.0f, be = 0.0f;
      if (hr == 1 && hr0 == 0) {  // computed during the first head's solve, already scanned
        g = s_G1[tid];
        be = s_beta1[tid];
      } else {
        if (tl < s_L[ci]) {
          if (hr == hr0)
            gate_log_raw(gr0, a.gate_mode, g, be);
          else
            gate_log(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                     static_cast<int64_t>(s_t0[ci] + tl) * a.Hv + h, h, g, be);
        }
        g = chunk_scan<C>(g, lane);
      }
      pad(tid, kBeta) = be;
      s_beta[tid] = be;
      s_G[tid] = g;
    }
    __syncthreads();
    if (C == 64 && tid >= 32 && tid < 64) s_G[tid] += s_G[31];  // read by all after the barrier below
    if (hr == hr0) {  // the G | QK product (issued once)
      if (!mbar_wait_bounded(bar, phase)) bad = true;
      bad = __any_sync(0xffffffffu, bad);
      phase ^= 1;
      tc::fence_after_sync();
    }
    __syncthreads();

    // A rows (warps on lanes 0..63, G) and P rows (warps on lanes 64..127, QK) from tensor
    // memory; thread: row t, column half `half`
    if (!bad) {
      const int q4 = warp & 3, half = warp >> 2;
      const bool is_p = q4 >= 2;
      const int t = 32 * (q4 & 1) + lane;
      const int ci = t / C, tl = t % C;
      const int c = c_first + ci;
      const bool live = c < nchunks && tl < s_L[ci];
      const float Gt = s_G[t];
      constexpr int NH = C / 2;  // columns per thread
      // tcgen05.ld is warp-collective with one column address per warp, so the
      // columns must not depend on the lane: for C >= 32 the warp's 32 rows lie
      // in one chunk; for C = 16 they span two chunks, both are loaded and each
      // lane keeps its own.
      float xv[NH];
      if constexpr (C >= 32) {
        const int cw = (32 * (q4 & 1)) / C;  // the warp's chunk
#pragma unroll
        for (int b0 = 0; b0 < NH; b0 += 16) {
          float tv[16];
          tmem_load<16>(tc::taddr(tb, 32 * q4, kColGQ + cw * C + half * NH + b0), tv);
#pragma unroll
          for (int e = 0; e < 16; ++e) xv[b0 + e] = tv[e];
        }
      } else {
        const int col0 = 32 * (q4 & 1) + half * NH;  // chunk 2q's half; +16: chunk 2q+1
        float xa[8], xb[8];
        tmem_load<8>(tc::taddr(tb, 32 * q4, kColGQ + col0), xa);
        tmem_load<8>(tc::taddr(tb, 32 * q4, kColGQ + col0 + 16), xb);
        const bool second = lane >= 16;
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] = second ? xb[e] : xa[e];
      }
      tc::tmem_wait_ld();
      if (!is_p) {
        const float bt = pad(t, kBeta), ikt = pad(t, kIk);
        float av[NH];
#pragma unroll
        for (int e4 = 0; e4 < NH; e4 += 4) {
          const int j0 = half * NH + e4, tj0 = ci * C + j0;
          const float4 G4 = *reinterpret_cast<const float4*>(s_G + tj0);
          const float4 K4 = *reinterpret_cast<const float4*>(s_ik + tj0);
          const float Gj[4] = {G4.x, G4.y, G4.z, G4.w}, ikj[4] = {K4.x, K4.y, K4.z, K4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = j0 + e;
            const float dec = (live && j < tl) ? __expf(Gt - Gj[e]) : 0.0f;
            av[e4 + e] = (j < tl) ? bt * dec * ikt * ikj[e] * xv[e4 + e] : 0.0f;
          }
        }
#pragma unroll
        for (int e = 0; e < NH; e += 4)  // the thread's half row of A, 16 bytes at a time
          *reinterpret_cast<float4*>(sA + t * SA + half * NH + e) =
              make_float4(av[e], av[e + 1], av[e + 2], av[e + 3]);
        // the token's W scale e^{G_t} ik_t (the solve reads columns 0 .. C-1 only)
        if (half == 0) s_bsc[t] = bt * (live ? expf(Gt) * ikt : 0.0f);
      } else if (c < nchunks) {
        const float iqt = pad(t, kIq) * a.scale;
        float pv[NH];
#pragma unroll
        for (int e4 = 0; e4 < NH; e4 += 4) {
          const int j0 = half * NH + e4, tj0 = ci * C + j0;
          const float4 G4 = *reinterpret_cast<const float4*>(s_G + tj0);
          const float4 K4 = *reinterpret_cast<const float4*>(s_ik + tj0);
          const float Gj[4] = {G4.x, G4.y, G4.z, G4.w}, ikj[4] = {K4.x, K4.y, K4.z, K4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = j0 + e;
            const float dec = (live && j <= tl) ? __expf(Gt - Gj[e]) : 0.0f;
            pv[e4 + e] = dec * iqt * ikj[e] * xv[e4 + e];
          }
        }
        unsigned char* ph = wb.Pt + (static_cast<size_t>(c) * a.Hv + h) * 2 * wb.p_tile;
#pragma unroll
        for (int e8 = 0; e8 < NH; e8 += 8) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = pv[e8 + e];
          uint4 hi, lo;
          split8(x, hi, lo);
          const uint32_t o = tc::kmajor_offset(tl, half * NH + e8, C);
          *reinterpret_cast<uint4*>(ph + o) = hi;
          *reinterpret_cast<uint4*>(ph + wb.p_tile + o) = lo;
        }
        if (half == 0) {
          float* vec = wb.vec + (static_cast<size_t>(c) * a.Hv + h) * kVecFloats;
          const float Glast = s_G[ci * C + max(s_L[ci] - 1, 0)];
          const float ikt = pad(t, kIk);
          vec[tl] = live ? expf(Gt) * iqt : 0.0f;               // f_t
          vec[64 + tl] = live ? expf(Glast - Gt) * ikt : 0.0f;  // dd_t
          if (tl == 0) vec[128] = expf(Glast);                  // g_last
        }
      }
    }
    bad = tc_sync(bad);
    if (bad) break;

    if (tid < kSolveThreads) {
      // exact fp32 T = (I + A)^-1 of every chunk, written over A in place (A is strictly lower
      // triangular, so its upper part already holds T's zeros), a blocked recursive inverse:
      // 1) the 8 x 8 diagonal blocks by forward substitution, a column per thread (threads
      //    0..63), A's rows read 16 bytes at a time (the same address across the block's threads)
      float x[8];
      const int R0 = 8 * (tid >> 3), cc = tid & 7;
      float* Ab = sA + R0 * SA + R0 % C;  // block entry (r, l): Ab[r * SA + l]
      if (tid < 64) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float4 a0 = *reinterpret_cast<const float4*>(Ab + r * SA);
          const float4 a1 = *reinterpret_cast<const float4*>(Ab + r * SA + 4);
          const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
          for (int l = 0; l < r; l += 2) {
            s0 = fmaf(av[l], x[l], s0);
            if (l + 1 < r) s1 = fmaf(av[l + 1], x[l + 1], s1);
          }
          x[r] = (r < cc) ? 0.0f : (r == cc ? 1.0f : -(s0 + s1));
        }
      }
      solver_sync();  // every diagonal block read
      if (tid < 64) {
#pragma unroll
        for (int r = 0; r < 8; ++r) Ab[r * SA + cc] = x[r];
      }
      // 2) blocks of 16, 32 and 64 rows, as far as the chunk goes, from their two halves
      solver_sync();
      solve_merge<8, C, SA>(sA, tid);
      if constexpr (C >= 32) {
        solver_sync();
        solve_merge<16, C, SA>(sA, tid);
      }
      if constexpr (C >= 64) {
        solver_sync();
        solve_merge<32, C, SA>(sA, tid);
      }
      solver_sync();
      // 3) T' = T diag(beta) and T'' = T diag(beta e^G ik) into the block-diagonal bf16 hi / lo
      //    tiles: row tid % 64, groups of 8 columns (tid / 64) + 2k, 16-byte stores (the warp's
      //    lanes on consecutive rows)
      {
        const int t = tid & 63, ci = t / C;
        const float* Tr = sA + t * SA;
        for (int g = tid >> 6; g < C / 8; g += 2) {
          const float4 u0 = *reinterpret_cast<const float4*>(Tr + 8 * g);
          const float4 u1 = *reinterpret_cast<const float4*>(Tr + 8 * g + 4);
          const float tv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          const int jb = ci * C + 8 * g;
          const float4 b0 = *reinterpret_cast<const float4*>(s_beta + jb);
          const float4 b1 = *reinterpret_cast<const float4*>(s_beta + jb + 4);
          const float4 c0 = *reinterpret_cast<const float4*>(s_bsc + jb);
          const float4 c1 = *reinterpret_cast<const float4*>(s_bsc + jb + 4);
          const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          float x1[8], x2[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x1[e] = tv[e] * bv[e];
            x2[e] = tv[e] * cv[e];
          }
          uint4 hi, lo;
          const uint32_t o = tc::kmajor_offset(t, jb, NR);
          split8(x1, hi, lo);
          *reinterpret_cast<uint4*>(sm + S::oT1h + o) = hi;
          *reinterpret_cast<uint4*>(sm + S::oT1l + o) = lo;
          split8(x2, hi, lo);
          *reinterpret_cast<uint4*>(sm + S::oT2h + o) = hi;
          *reinterpret_cast<uint4*>(sm + S::oT2l + o) = lo;
        }
      }
    } else {
      // V (raw bf16) as an MN-major operand over the 64 tokens, in the k tile's layout:
      // 16-byte pieces of 8 channels of one token. A thread takes channel group cg of tokens
      // 8i + (u & 7), i = 0..7: the 8 lanes sharing cg hold 8 consecutive tokens, so each
      // 16-byte store hits its own bank group. All 8 loads are issued before the first store
      const int u = tid - kSolveThreads;
      const int cg = (u >> 3) & 15, tr = u & 7;
      const uint16_t* yv = y + 2 * a.Hk * kD + h * kD + 8 * cg;
      uint4 vb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int tok = 8 * i + tr, ci = tok / C, tl = tok % C;
        vb[i] = tl < s_L[ci]
                    ? __ldg(reinterpret_cast<const uint4*>(yv + static_cast<int64_t>(s_t0[ci] + tl) * a.D))
                    : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        *reinterpret_cast<uint4*>(sm + S::oV + tc::kmajor_offset(8 * i + tr, 8 * cg, kD)) = vb[i];
      // then, for the first value head, the q and k tiles of each chunk -> workspace (a
      // chunk's rows are one contiguous slice of either smem tile)
      for (int ci = 0; ci < CPC && hr == 0; ++ci) {
        const int c = c_first + ci;
        if (c >= nchunks) break;
        const size_t slice = static_cast<size_t>(C) * kD * 2;  // bytes of one chunk's tile
        const uint4* srcq = reinterpret_cast<const uint4*>(sm + S::oQ + ci * slice);
        const uint4* srck = reinterpret_cast<const uint4*>(sm + S::oK + ci * slice);
        uint4* dq = reinterpret_cast<uint4*>(wb.Qt + (static_cast<size_t>(c) * a.Hk + kh) * wb.q_tile);
        uint4* dk = reinterpret_cast<uint4*>(wb.Kt + (static_cast<size_t>(c) * a.Hk + kh) * wb.q_tile);
        for (int i = u; i < static_cast<int>(slice / 16); i += kThreadsTc - kSolveThreads) {
          dq[i] = srcq[i];
          dk[i] = srck[i];
        }
      }
      // then, during the first head's solve, the second head's gates (warps 4 and 5, token row
      // u), scanned within the warp as that head's gate phase would
      if (hr == 0 && hr1 > 1 && u < NR) {
        const int ci = u / C, tl = u % C, h1 = kh * R + 1;
        float g = 0.0f, be = 0.0f;
        if (tl < s_L[ci])
          gate_log(a.a, a.b, a.gate_mode, a.A_log, a.dt_bias,
                   static_cast<int64_t>(s_t0[ci] + tl) * a.Hv + h1, h1, g, be);
        s_G1[u] = chunk_scan<C>(g, lane);
        s_beta1[u] = be;
      }
    }
    bad = tc_sync(bad);
    if (bad) break;

    if (tid == 0) {
      // U^T = V^T T'^T (a dv row per lane, a token per column), A = V MN-major;
      // W = T'' K (a token per lane), B = K MN-major
      const uint32_t idu = tc::idesc_bf16_f32_amn(128, NR);
      const uint32_t idw = tc::idesc_bf16_f32_bmn(128, kD);
      const uint32_t t1h = smem_addr(sm + S::oT1h), t1l = smem_addr(sm + S::oT1l);
      const uint32_t t2h = smem_addr(sm + S::oT2h), t2l = smem_addr(sm + S::oT2l);
      const uint32_t v = smem_addr(sm + S::oV), k = smem_addr(sm + S::oK);
      constexpr int KS = NR / 16;
      for (int ks = 0; ks < KS; ++ks)
        tc::mma_bf16(tb + kColU, tc::mnmajor_desc(v, kD, ks), tc::kmajor_desc(t1h, NR, ks), idu, ks > 0);
      for (int ks = 0; ks < KS; ++ks)
        tc::mma_bf16(tb + kColU, tc::mnmajor_desc(v, kD, ks), tc::kmajor_desc(t1l, NR, ks), idu, 1);
      for (int ks = 0; ks < KS; ++ks)
        tc::mma_bf16(tb + kColW, tc::kmajor_desc(t2h, NR, ks), tc::mnmajor_desc(k, kD, ks), idw, ks > 0);
      for (int ks = 0; ks < KS; ++ks)
        tc::mma_bf16(tb + kColW, tc::kmajor_desc(t2l, NR, ks), tc::mnmajor_desc(k, kD, ks), idw, 1);
      tc::mma_commit(bar);
    }
    if (!mbar_wait_bounded(bar, phase)) bad = true;
    bad = __any_sync(0xffffffffu, bad);  // warp-uniform before the aligned loads
    phase ^= 1;
    tc::fence_after_sync();
    if (!bad) {
      // U^T -> workspace (fp32 [128 x C] tile image per chunk, 16-byte pieces of a dv row):
      // every warp, lane = dv row r, 32 token columns per warp
      const int r = 32 * (warp & 3) + lane, half = warp >> 2;
      {
        float uv[32];
        tmem_load<16>(tc::taddr(tb, 32 * (warp & 3), kColU + half * 32),
                      *reinterpret_cast<float(*)[16]>(uv));
        tmem_load<16>(tc::taddr(tb, 32 * (warp & 3), kColU + half * 32 + 16),
                      *reinterpret_cast<float(*)[16]>(uv + 16));
        tc::tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < 32; g += 8) {  // 8 tokens of one chunk: two 16-byte image pieces
          const int T = half * 32 + g, cu = c_first + T / C, tu = T % C;
          if (cu < nchunks) {
            unsigned char* ub = reinterpret_cast<unsigned char*>(
                wb.Ut + (static_cast<size_t>(cu) * a.Hv + h) * (kD * C));
            *reinterpret_cast<float4*>(ub + u_image_offset(r, tu, C)) =
                make_float4(uv[g], uv[g + 1], uv[g + 2], uv[g + 3]);
            *reinterpret_cast<float4*>(ub + u_image_offset(r, tu + 4, C)) =
                make_float4(uv[g + 4], uv[g + 5], uv[g + 6], uv[g + 7]);
          }
        }
      }
      // W -> hi / lo tiles [C x 128]: warps whose lanes hold token rows 0..63, lane = token
      // row t, 64 columns per warp. Every lane of such a warp executes the (warp-collective)
      // loads; only existing chunks store
      if ((warp & 3) < 2) {
        const int t = r, ci = t / C, tl = t % C, c = c_first + ci;
        const bool store = c < nchunks;
        unsigned char* wt = wb.Wt + (static_cast<size_t>(store ? c : 0) * a.Hv + h) * 2 * wb.w_tile;
#pragma unroll 1
        for (int b0 = 0; b0 < 64; b0 += 16) {
          const int col = half * 64 + b0;
          float wv[16];
          tmem_load<16>(tc::taddr(tb, 32 * (warp & 3), kColW + col), wv);  // W[t][col ..]
          tc::tmem_wait_ld();
          if (!store) continue;
#pragma unroll
          for (int e8 = 0; e8 < 16; e8 += 8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = wv[e8 + e];
            uint4 hi, lo;
            split8(x, hi, lo);
            const uint32_t o = tc::kmajor_offset(tl, col + e8, 128);
            *reinterpret_cast<uint4*>(wt + o) = hi;
            *reinterpret_cast<uint4*>(wt + wb.w_tile + o) = lo;
          }
        }
      }
    }
    bad = tc_sync(bad);
  }
  if (bad && tid == 0 && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
  tc_sync(false);
  if (warp == 0) tc::tmem_dealloc(tb, kIntraTmemCols);
  grid_dep_launch();
  if (waits) grid_dep_wait();
}

// ============================================================== pass kernel
template <int C>
struct PassSmem {
  static constexpr int kUh = 128 * C * 2;       // one half of the U^T image (u_image_offset)
  static constexpr int kW = C * 128 * 2;        // W, Q tiles [C x 128]   bf16
  static constexpr int kP = C * C * 2;          // P tiles    [C x C]     bf16
  static constexpr int oU = 0;                  // U^T image, fp32 [128 x C]: 2 kUh bytes
  // the q tile follows the W hi tile: together they are one [2C x 128] MMA operand
  static constexpr int oWh = oU + 2 * kUh, oQ = oWh + kW, oWl = oQ + kW;
  static constexpr int oPh = oWl + kW, oPl = oPh + kP, oKtile = oPl + kP;  // k tile [C x 128]
  static constexpr int oVec = oKtile + kW;      // two vec buffers of kVecFloats
  static constexpr int oO = oVec + 2 * kVecFloats * 4;  // bf16 output tile [C x 128], swizzled
  static constexpr int kBytes = oO + C * 128 * 2;
  // the kernel's static variables (tensor-memory base, mbarriers) are padded to 1 KB ahead of
  // the 1 KB-aligned dynamic block
  static_assert(kBytes + 1024 <= 227 * 1024, "pass shared memory exceeds the per-CTA limit");
};

template <int C>
__global__ void __launch_bounds__(kPassThreads, 1)
    pass_tc_kernel(LayerArgs a, PrefillExtra p, const int32_t* seq_ok, const int32_t* chunk_off,
                   const int32_t* seq_order, TcBufs wb, int g_lo, int g_hi, float* sx, int pdl) {
  // [g_lo, g_hi): the chunks of this launch (a piece of the call's chunks, or all of them); a
  // sequence's state enters from its slot at its first chunk, else from sx, and leaves to its
  // slot after its last chunk, else to sx. pdl: launched as a programmatic dependent of the
  // piece's intra kernel (which follows the pass over the piece before)
  using S = PassSmem<C>;
  // the next piece's intra kernel may start once every CTA of this pass is resident
  if (pdl) grid_dep_launch();
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ uint32_t s_tmem;
  // fullA, fullB, mma1, mma2, fullU, oDone, dead, upd, scaled
  __shared__ __align__(8) uint64_t s_bar[9];

  // CTAs in launch order take the sequences longest first, all value heads of one together
  const int i = seq_order[blockIdx.x / a.Hv], h = blockIdx.x % a.Hv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bos = p.cu_seqlens[i], eos = p.cu_seqlens[i + 1];
  if (!seq_ok[i]) {  // inactive / invalid sequence (or bad cu_seqlens): zero outputs, once
    if (g_lo != 0) return;
    int64_t n = static_cast<int64_t>(max(eos - bos, 0));
    if (bos < 0 || eos > p.total_tokens) n = 0;
    for (int64_t idx = tid; idx < n * kD; idx += kPassThreads) {
      const int64_t o = ((bos + idx / kD) * a.Hv + h) * kD + idx % kD;
      if (a.out_f32) static_cast<float*>(a.out)[o] = 0.0f;
      else static_cast<uint16_t*>(a.out)[o] = 0;
    }
    return;
  }
  const int cs = chunk_off[i], ce = chunk_off[i + 1];  // the sequence's chunks
  int c0 = cs, c1 = ce;  // this launch's share of them: [c0, c1)
  if (cs == ce) {        // no token: the first piece stores the initial (or zero) state
    if (g_lo != 0) return;
  } else {
    c0 = max(cs, g_lo);
    c1 = min(ce, g_hi);
    if (c1 <= c0) return;
  }
  const int nch = c1 - c0;
  const bool from_slot = c0 == cs, to_slot = c1 == ce;
  // tensor memory first: no return follows, and no other CTA that uses it shares this SM (shared
  // memory excludes the intra kernel's), so the allocation does not wait on the kernels before
  if (warp == 0) tc::tmem_alloc(&s_tmem, kTmemCols);
  if (pdl) grid_dep_wait();  // the piece's intra tiles, and the state the piece before left in sx
  const int32_t slot = a.slot[i];
  const bool init = (p.has_init == nullptr) || (p.has_init[i] != 0);
  const bool mma_warp = warp == kThreadsTc / 32, copy_warp = warp == kThreadsTc / 32 + 1;
  const bool compute = warp < kThreadsTc / 32;
  const int q = warp & 3, half = warp >> 2;  // compute warps
  const int r = 32 * q + lane;  // state row (dv index) = tensor-memory lane
  // Tensor-memory columns. X0 = [0, 128) and X1 = [256, 384) alternate by chunk parity p:
  // chunk it's raw D^T (then its O2^T) at [X_p, X_p + C) and O1^T at [X_p + C, X_p + 2C), its
  // state update at [X_(1-p), X_(1-p) + 128) -- free by then, the chunk before's output has
  // been read. The A operands of the MMAs (bf16 pairs of K per column): the state's hi / lo
  // parts at [kColS, kColS + 64) / [kColS + 64, kColS + 128), D^T hi / lo and D'^T hi / lo at
  // kColDE + {0, C / 2, C, 3C / 2}, C / 2 columns each.
  constexpr int kColS = 128, kColDE = 384;
  const uint32_t fullA = smem_addr(&s_bar[0]), fullB = smem_addr(&s_bar[1]);
  const uint32_t mma1 = smem_addr(&s_bar[2]), mma2 = smem_addr(&s_bar[3]);
  const uint32_t fullU = smem_addr(&s_bar[4]);
  // oDone: every compute warp has finished chunk it's output (and with vec[it & 1]); the
  // copy warp's own arrival for a phase comes only after it has seen the one before, so
  // no warp's arrivals can run into the next phase
  const uint32_t oDone = smem_addr(&s_bar[5]);
  const uint32_t dead = smem_addr(&s_bar[6]);  // never arrived on (test hook)
  // group 2 is committed in two parts: upd once the state update D'^T K is done (all the
  // state chain waits for), mma2 once O2^T = D^T P^T is done too (the output, and the reuse of
  // the P, k and U buffers, wait for that)
  const uint32_t upd = smem_addr(&s_bar[7]);
  // scaled: every compute warp has replaced its O1 columns by f_t O1 (one arrival per warp),
  // on which the O2 products then accumulate
  const uint32_t scaled = smem_addr(&s_bar[8]);
  const int test_fault = g_test_fault;
  const size_t wtile = wb.w_tile, ptile = wb.p_tile;

  // W hi/lo, q tile, vec of chunk c0 + it on one fullA phase (group 1's operands, and vec)
  auto issue_A = [&](int it) {
    const int c = c0 + it;
    const int kh = h / (a.Hv / a.Hk);
    const unsigned char* w = wb.Wt + (static_cast<size_t>(c) * a.Hv + h) * 2 * wtile;
    const unsigned char* qt = wb.Qt + (static_cast<size_t>(c) * a.Hk + kh) * wb.q_tile;
    const float* vec = wb.vec + (static_cast<size_t>(c) * a.Hv + h) * kVecFloats;
    mbar_arrive_expect_tx(fullA, static_cast<uint32_t>(2 * wtile + wb.q_tile + kVecFloats * 4));
    bulk_g2s(smem_addr(sm + S::oWh), w, static_cast<uint32_t>(wtile), fullA);
    bulk_g2s(smem_addr(sm + S::oWl), w + wtile, static_cast<uint32_t>(wtile), fullA);
    bulk_g2s(smem_addr(sm + S::oQ), qt, static_cast<uint32_t>(wb.q_tile), fullA);
    bulk_g2s(smem_addr(sm + S::oVec + (it & 1) * kVecFloats * 4), vec, kVecFloats * 4, fullA);
  };
  auto issue_B = [&](int it) {  // P hi/lo, k tile of chunk c0 + it
    const int c = c0 + it;
    const int kh = h / (a.Hv / a.Hk);
    const unsigned char* pp = wb.Pt + (static_cast<size_t>(c) * a.Hv + h) * 2 * ptile;
    const unsigned char* kt = wb.Kt + (static_cast<size_t>(c) * a.Hk + kh) * wb.q_tile;
    mbar_arrive_expect_tx(fullB, static_cast<uint32_t>(2 * ptile + wb.q_tile));
    bulk_g2s(smem_addr(sm + S::oPh), pp, static_cast<uint32_t>(ptile), fullB);
    bulk_g2s(smem_addr(sm + S::oPl), pp + ptile, static_cast<uint32_t>(ptile), fullB);
    bulk_g2s(smem_addr(sm + S::oKtile), kt, static_cast<uint32_t>(wb.q_tile), fullB);
  };
  auto issue_U = [&](int it) {  // U^T of chunk c0 + it (its buffer is free once group 2 is done)
    const float* ut = wb.Ut + (static_cast<size_t>(c0 + it) * a.Hv + h) * (kD * C);
    mbar_arrive_expect_tx(fullU, static_cast<uint32_t>(kD * C * 4));
    bulk_g2s(smem_addr(sm + S::oU), ut, static_cast<uint32_t>(kD * C * 4), fullU);
  };

  if (copy_warp && lane == 0) {
    for (int k = 0; k < 5; ++k) mbar_init(smem_addr(&s_bar[k]), 1);
    mbar_init(dead, 1);
    mbar_init(upd, 1);
    mbar_init(scaled, kThreadsTc / 32);
    mbar_init(oDone, kThreadsTc / 32 + 1);
    fence_mbar_init();
    if (nch > 0) { issue_A(0); issue_B(0); issue_U(0); }
  }
  // state (half a row per compute thread) -> registers; its split parts -> tensor memory below
  const int64_t soff = (static_cast<int64_t>(slot) * a.Hv + h) * (kD * kD) + r * kD + half * 64;
  float* Sg = a.ssm + soff;                                          // fp32 state
  uint16_t* Sb = reinterpret_cast<uint16_t*>(a.ssm) + soff;          // bf16 state
  // the state between pieces: per (sequence, value head) 64 KB of fp32, float4 piece j of row r at
  // [j][r] (j = 0 .. 31 along dk), so that a warp's 32 rows read or write 512 contiguous bytes
  float* Sx = sx ? sx + (static_cast<int64_t>(i) * a.Hv + h) * (kD * kD) + (half * 16 * 128 + r) * 4
                 : nullptr;
  float Sr[64];
  if (compute && !from_slot) {
#pragma unroll
    for (int e = 0; e < 64; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(Sx + e / 4 * 128 * 4);
      Sr[e] = v.x; Sr[e + 1] = v.y; Sr[e + 2] = v.z; Sr[e + 3] = v.w;
    }
  } else if (compute) {
    if (a.ssm_bf16) {
#pragma unroll
      for (int e = 0; e < 64; e += 8) {
        float f[8];
        unpack8(init ? *reinterpret_cast<const uint4*>(Sb + e) : make_uint4(0u, 0u, 0u, 0u), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) Sr[e + i] = f[i];
      }
    } else {
#pragma unroll
      for (int e = 0; e < 64; e += 4) {
        float4 v = init ? *reinterpret_cast<const float4*>(Sg + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        Sr[e] = v.x; Sr[e + 1] = v.y; Sr[e + 2] = v.z; Sr[e + 3] = v.w;
      }
    }
  }
  tc_sync(false);  // the tensor-memory allocation is visible
  const uint32_t tb = s_tmem;
  // the state's bf16 hi / lo parts, the A operand of group 1, in tensor memory: this thread's
  // half row r, 32 columns of k pairs each
  auto store_S_tmem = [&]() {
#pragma unroll
    for (int e8 = 0; e8 < 64; e8 += 8) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = Sr[e8 + e];
      uint4 hi, lo;
      split8(x, hi, lo);
      const int col = half * 32 + e8 / 2;
      tc::tmem_st4(tc::taddr(tb, 32 * q, kColS + col), hi);
      tc::tmem_st4(tc::taddr(tb, 32 * q, kColS + 64 + col), lo);
    }
    tc::tmem_wait_st();
  };
  if (compute) store_S_tmem();
  bool bad = tc_sync(false);
  bool mine = false;  // this thread's wait failure, reported at the next CTA barrier
  constexpr int NH = C / 2;
  constexpr int KS = C / 16;
  // operand descriptors are fixed per CTA; a K step adds 256 bytes (16 units) to the start
  const uint64_t dWh = tc::kmajor_desc(smem_addr(sm + S::oWh), 128, 0);
  const uint64_t dWl = tc::kmajor_desc(smem_addr(sm + S::oWl), 128, 0);
  const uint64_t dPh = tc::kmajor_desc(smem_addr(sm + S::oPh), C, 0);
  const uint64_t dPl = tc::kmajor_desc(smem_addr(sm + S::oPl), C, 0);
  const uint64_t dKtile = tc::mnmajor_desc(smem_addr(sm + S::oKtile), 128, 0);  // k tile, MN-major
  const uint32_t idC = tc::idesc_bf16_f32(128, C), id2C = tc::idesc_bf16_f32(128, 2 * C);
  const uint32_t id128m = tc::idesc_bf16_f32_bmn(128, 128);

  // MMA group 1 of chunk `it` (the MMA warp): S [W_hi | Q]^T over N = 2C puts S W_hi^T into
  // the D^T columns and S Q^T (= O1^T, both S parts) into the next C; S_hi W_lo^T completes D
  auto issue_mma1 = [&](int it) -> bool {
    if (!mbar_wait_bounded(fullA, it & 1)) return false;
    const uint32_t t1 = tb + ((it & 1) ? 256 : 0);
    const uint32_t aSh = tb + kColS, aSl = tb + kColS + 64;  // a K step: 8 columns
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) tc::mma_bf16_ts(t1, aSh + 8 * ks, dWh + 16 * ks, id2C, ks > 0);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) tc::mma_bf16_ts(t1, aSl + 8 * ks, dWh + 16 * ks, id2C, 1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) tc::mma_bf16_ts(t1, aSh + 8 * ks, dWl + 16 * ks, idC, 1);
    tc::mma_commit(mma1);
    return true;
  };
  // an MMA-warp failure leaves an MMA group unissued; the compute threads' bounded waits
  // then expire, and every thread learns of it at the next barrier
  if (mma_warp && lane == 0 && nch > 0 && !bad) mine = !issue_mma1(0);

  auto prefetch_chunk = [&](int it) {  // the workspace tiles of chunk c0 + it -> L2
    const int c = c0 + it;
    const int kh = h / (a.Hv / a.Hk);
    const size_t ch = static_cast<size_t>(c) * a.Hv + h;
    bulk_prefetch_l2(wb.Ut + ch * (kD * C), static_cast<uint32_t>(kD * C * 4));
    bulk_prefetch_l2(wb.Wt + ch * 2 * wtile, static_cast<uint32_t>(2 * wtile));
    bulk_prefetch_l2(wb.Pt + ch * 2 * ptile, static_cast<uint32_t>(2 * ptile));
    bulk_prefetch_l2(wb.vec + ch * kVecFloats, kVecFloats * 4);
    const size_t ck = static_cast<size_t>(c) * a.Hk + kh;
    bulk_prefetch_l2(wb.Qt + ck * wb.q_tile, static_cast<uint32_t>(wb.q_tile));
    bulk_prefetch_l2(wb.Kt + ck * wb.q_tile, static_cast<uint32_t>(wb.q_tile));
  };
  if (copy_warp) {
    // each chunk's tiles as soon as their buffers are free: P, k and U of chunk it + 1 once
    // group 2 of chunk it is done (and so the D phase that read U); W, q and vec of chunk it + 2
    // once group 1 of chunk it + 1 is done and every compute warp has finished chunk it's
    // output (vec[it & 1]). Each barrier of a chunk is armed only after this warp has seen
    // the phase it waits on for the chunk before, so no parity wait can alias a later phase
    bool ok = !bad;
    if (lane == 0 && nch > 0) {
      int nA = 1, nBU = 1;  // phases issued (chunk 0's at set-up)
      if (nch > 1) prefetch_chunk(1);
      mbar_arrive(oDone);  // this warp's share of phase 0
      if (ok && nch > 1) {
        if (mbar_wait_bounded(mma1, 0)) {
          tc::fence_after_sync();
          issue_A(1);
          nA = 2;
        } else {
          ok = false;
        }
      }
      for (int it = 0; ok && it + 1 < nch; ++it) {
        const uint32_t par = it & 1;
        if (it + 2 < nch) prefetch_chunk(it + 2);  // two chunks ahead
        if (!mbar_wait_bounded(mma2, par)) { ok = false; break; }
        tc::fence_after_sync();
        issue_B(it + 1);
        issue_U(it + 1);
        nBU = it + 2;
        if (it + 2 < nch) {
          if (!mbar_wait_bounded(oDone, par)) { ok = false; break; }
          mbar_arrive(oDone);  // share of phase it + 1
          if (!mbar_wait_bounded(mma1, par ^ 1)) { ok = false; break; }
          tc::fence_after_sync();
          issue_A(it + 2);
          nA = it + 3;
        }
      }
      if (!ok && a.err) atomicOr(a.err, GDN_DEVERR_TIMEOUT);
      // copies may still be in flight -- after this warp's own failure, and after another
      // warp's, which leaves the chunk loop without waiting for the tiles already issued for
      // the next chunk: wait (bounded) for the last issued phase of each barrier before the
      // CTA may exit; one already completed (and consumed) returns at once
      mbar_wait_bounded(fullA, (nA - 1) & 1);
      mbar_wait_bounded(fullB, (nBU - 1) & 1);
      mbar_wait_bounded(fullU, (nBU - 1) & 1);
    }
  }

  int n1 = (mma_warp && nch > 0 && !mine) ? 1 : 0, n2 = 0;  // MMA groups committed
  for (int it = 0; it < nch && !bad && !copy_warp; ++it) {
    const int t0 = bos + (c0 - cs + it) * C;
    const int L = min(C, eos - t0);
    const uint32_t par = it & 1;
    const float* vec = reinterpret_cast<const float*>(sm + S::oVec + par * kVecFloats * 4);
    const int base = par ? 256 : 0, other = par ? 0 : 256;  // X_p, X_(1-p)
    if (compute) {
      if (!mbar_wait_bounded(mma1, par)) mine = true;
      if (!mbar_wait_bounded(fullU, par)) mine = true;
      mine = __any_sync(0xffffffffu, mine);  // warp-uniform before the aligned loads
      tc::fence_after_sync();
      if (!mine) {
        // D = U - raw, D' = D dd_t; both split into the [128 x C] operand tiles
        float raw[NH];
        if constexpr (NH >= 16) {
#pragma unroll
          for (int b0 = 0; b0 < NH; b0 += 16) {
            float tv[16];
            tmem_load<16>(tc::taddr(tb, 32 * q, base + half * NH + b0), tv);
#pragma unroll
            for (int e = 0; e < 16; ++e) raw[b0 + e] = tv[e];
          }
        } else {
          float tv[8];
          tmem_load<8>(tc::taddr(tb, 32 * q, base + half * NH), tv);
#pragma unroll
          for (int e = 0; e < 8; ++e) raw[e] = tv[e];
        }
        tc::tmem_wait_ld();
#pragma unroll
        for (int e8 = 0; e8 < NH; e8 += 8) {
          const uint32_t o = tc::kmajor_offset(r, half * NH + e8, C);
          // this thread's U^T values of the 8 tokens (two 16-byte pieces of the image)
          const float4 u0 = *reinterpret_cast<const float4*>(sm + S::oU + o);
          const float4 u1 = *reinterpret_cast<const float4*>(sm + S::oU + S::kUh + o);
          const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          float d[8], dd[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            d[e] = u[e] - raw[e8 + e];
            dd[e] = d[e] * vec[64 + half * NH + e8 + e];
          }
          uint4 hi, lo;
          const int col = kColDE + (half * NH + e8) / 2;  // token pairs of row r
          split8(d, hi, lo);
          tc::tmem_st4(tc::taddr(tb, 32 * q, col), hi);
          tc::tmem_st4(tc::taddr(tb, 32 * q, col + C / 2), lo);
          split8(dd, hi, lo);
          tc::tmem_st4(tc::taddr(tb, 32 * q, col + C), hi);
          tc::tmem_st4(tc::taddr(tb, 32 * q, col + 3 * C / 2), lo);
        }
        tc::tmem_wait_st();
      }
    }
    bad = pass_sync(mine);
    if (bad) break;
    if (mma_warp) {
      // ---- MMA group 2: O2^T = D^T P^T (3 products), update = D'^T K (2 products)
      if (lane == 0) {
        if (mbar_wait_bounded(fullB, par)) {
          // the update into X_(1-p) first (the state chain waits for it alone), then O2^T over
          // the raw D^T columns (read by now); A operands from tensor memory, a K step of 8
          // columns
          const uint32_t aDh = tb + kColDE, aDl = aDh + C / 2, aEh = aDh + C, aEl = aDh + 3 * C / 2;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)  // a K step of the MN-major k tile: 4096 bytes (256 units)
            tc::mma_bf16_ts(tb + other, aEh + 8 * ks, dKtile + 256 * ks, id128m, ks > 0);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
            tc::mma_bf16_ts(tb + other, aEl + 8 * ks, dKtile + 256 * ks, id128m, 1);
          tc::mma_commit(upd);
          // O = f_t O1 + O2: the O2 products accumulate onto the O1 columns once every compute
          // warp has scaled them (committed whatever happened, so that what was issued can be
          // waited for)
          if (mbar_wait_bounded(scaled, par)) {
            tc::fence_after_sync();
            const uint32_t tO = tb + base + C;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) tc::mma_bf16_ts(tO, aDh + 8 * ks, dPh + 16 * ks, idC, 1);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) tc::mma_bf16_ts(tO, aDh + 8 * ks, dPl + 16 * ks, idC, 1);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) tc::mma_bf16_ts(tO, aDl + 8 * ks, dPh + 16 * ks, idC, 1);
          } else {
            mine = true;
          }
          tc::mma_commit(mma2);
          n2 = it + 1;
        } else {
          mine = true;
        }
      }
    } else {  // compute warps
      {
        // f_t O1 in place over this thread's O1 columns, while the state update runs; the O2
        // products then accumulate onto it. (No wait failed before the barrier, or the loop
        // would have ended.)
        float o1[NH];
        if constexpr (NH >= 16) {
#pragma unroll
          for (int b0 = 0; b0 < NH; b0 += 16) {
            float tv[16];
            tmem_load<16>(tc::taddr(tb, 32 * q, base + C + half * NH + b0), tv);
#pragma unroll
            for (int e = 0; e < 16; ++e) o1[b0 + e] = tv[e];
          }
        } else {
          float tv[8];
          tmem_load<8>(tc::taddr(tb, 32 * q, base + C + half * NH), tv);
#pragma unroll
          for (int e = 0; e < 8; ++e) o1[e] = tv[e];
        }
        tc::tmem_wait_ld();
        if constexpr (NH >= 16) {
#pragma unroll
          for (int b0 = 0; b0 < NH; b0 += 16) {
            float tv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) tv[e] = vec[half * NH + b0 + e] * o1[b0 + e];
            tc::tmem_st16(tc::taddr(tb, 32 * q, base + C + half * NH + b0), tv);
          }
        } else {
          float tv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) tv[e] = vec[half * NH + e] * o1[e];
          tc::tmem_st8(tc::taddr(tb, 32 * q, base + C + half * NH), tv);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(scaled);
      }
      const bool test_fail = test_fault == 2 && blockIdx.x == 0 && warp == 0 && it == 0;
      if (test_fail ? !mbar_wait_bounded(dead, 0, kTestWaitNs) : !mbar_wait_bounded(upd, par))
        mine = true;
      mine = __any_sync(0xffffffffu, mine);  // warp-uniform before the aligned loads
      tc::fence_after_sync();
      if (!mine) {
        // S <- g_last S + update, 16 columns at a time
        const float gl = vec[128];
#pragma unroll
        for (int b0 = 0; b0 < 64; b0 += 32) {  // two loads in flight per wait
          float tv0[16], tv1[16];
          tmem_load<16>(tc::taddr(tb, 32 * q, other + half * 64 + b0), tv0);
          tmem_load<16>(tc::taddr(tb, 32 * q, other + half * 64 + b0 + 16), tv1);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            Sr[b0 + e] = fmaf(gl, Sr[b0 + e], tv0[e]);
            Sr[b0 + 16 + e] = fmaf(gl, Sr[b0 + 16 + e], tv1[e]);
          }
        }
        store_S_tmem();
      }
    }
    bad = pass_sync(mine);
    if (bad) break;
    if (mma_warp) {
      if (lane == 0 && it + 1 < nch) {
        mine = !issue_mma1(it + 1);
        if (!mine) n1 = it + 2;
      }
    } else {
      // chunk it's output O = f_t O1 + O2 (formed by group 2 in the O1 columns), while group 1
      // of chunk it + 1 runs (O is there once the whole of group 2 is done; a failed wait
      // skips the output)
      if (!mbar_wait_bounded(mma2, par)) mine = true;
      mine = __any_sync(0xffffffffu, mine);  // warp-uniform before the aligned loads
      tc::fence_after_sync();
      if (!mine) {
        float ov[NH];
        if constexpr (NH >= 16) {
#pragma unroll
          for (int b0 = 0; b0 < NH; b0 += 16) {
            float ta[16];
            tmem_load<16>(tc::taddr(tb, 32 * q, base + C + half * NH + b0), ta);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[b0 + e] = ta[e];
          }
        } else {
          float ta[8];
          tmem_load<8>(tc::taddr(tb, 32 * q, base + C + half * NH), ta);
#pragma unroll
          for (int e = 0; e < 8; ++e) ov[e] = ta[e];
        }
        tc::tmem_wait_ld();
        if (a.out_f32) {
#pragma unroll
          for (int e = 0; e < NH; ++e) {
            const int tt = half * NH + e;
            if (tt < L)
              static_cast<float*>(a.out)[(static_cast<int64_t>(t0 + tt) * a.Hv + h) * kD + r] = ov[e];
          }
        } else {
          // stage the warp's [NH tokens x 32 dv] block in the bf16 tile, then copy it out in
          // 16-byte pieces; the tile's 16-byte pieces are XOR-swizzled by token so both the
          // 2-byte writes and the 16-byte reads are free of bank conflicts
          unsigned char* ot = sm + S::oO;
#pragma unroll
          for (int e = 0; e < NH; ++e) {
            const int tt = half * NH + e;
            *reinterpret_cast<uint16_t*>(ot + out_tile_offset(tt, r)) = f2bf(ov[e]);
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < NH / 8; ++k) {
            const int pc = lane + 32 * k;
            const int tt = half * NH + pc / 4, col = 32 * q + (pc % 4) * 8;
            if (tt < L)
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) +
                                        (static_cast<int64_t>(t0 + tt) * a.Hv + h) * kD + col) =
                  *reinterpret_cast<const uint4*>(ot + out_tile_offset(tt, col));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(oDone);  // this warp is done with chunk it's output and vec
    }
  }
  if (!copy_warp) bad = pass_sync(bad || mine);
  if (bad && mma_warp && lane == 0) {
    // after a failure, let the committed MMA groups finish before tensor memory is freed
    if (n1 > 0) mbar_wait_bounded(mma1, (n1 - 1) & 1);
    if (n2 > 0) mbar_wait_bounded(mma2, (n2 - 1) & 1);
  }
  if (!bad) {
    if (compute && !to_slot) {  // the next piece takes the state from here, unrounded
#pragma unroll
      for (int e = 0; e < 64; e += 4)
        *reinterpret_cast<float4*>(Sx + e / 4 * 128 * 4) = make_float4(Sr[e], Sr[e + 1], Sr[e + 2], Sr[e + 3]);
    } else if (compute) {
      if (a.ssm_bf16) {  // rounded to bf16 only here, at the write-back
#pragma unroll
        for (int e = 0; e < 64; e += 8) {
          uint16_t hb[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) hb[i] = f2bf(Sr[e + i]);
          *reinterpret_cast<uint4*>(Sb + e) = pack8(hb);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 64; e += 4)
          *reinterpret_cast<float4*>(Sg + e) = make_float4(Sr[e], Sr[e + 1], Sr[e + 2], Sr[e + 3]);
      }
    }
  } else if (tid == 0 && a.err) {
    atomicOr(a.err, GDN_DEVERR_TIMEOUT);
  }
  tc_sync(false);
  if (warp == 0) tc::tmem_dealloc(tb, kTmemCols);
}

// A kernel launch, as a programmatic dependent of the stream's previous kernel when `pdl`.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t s,
                     bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int C>
cudaError_t launch_tc_c(const LayerArgs& a, const PrefillExtra& p, const TcLayout& L, char* ws,
                        const uint16_t* y, cudaStream_t s) {
  const int32_t* meta = reinterpret_cast<const int32_t*>(ws + L.meta);
  const int32_t* seq_ok = reinterpret_cast<const int32_t*>(ws + L.seq_ok);
  const int32_t* chunk_off = reinterpret_cast<const int32_t*>(ws + L.chunk_off);
  const int32_t* chunk_seq = reinterpret_cast<const int32_t*>(ws + L.chunk_seq);
  const int32_t* seq_order = reinterpret_cast<const int32_t*>(ws + L.seq_order);
  TcBufs wb;
  wb.Qt = reinterpret_cast<unsigned char*>(ws + L.Qt);
  wb.Kt = reinterpret_cast<unsigned char*>(ws + L.Kt);
  wb.Wt = reinterpret_cast<unsigned char*>(ws + L.Wt);
  wb.Pt = reinterpret_cast<unsigned char*>(ws + L.Pt);
  wb.Ut = reinterpret_cast<float*>(ws + L.Ut);
  wb.vec = reinterpret_cast<float*>(ws + L.vec);
  wb.q_tile = L.q_tile;
  wb.w_tile = L.w_tile;
  wb.p_tile = L.p_tile;
  constexpr int CPC = IntraSmem<C>::CPC;
  const int M = L.max_chunks;  // an upper bound of the call's chunks
  auto k1 = intra_tc_kernel<C>;
  auto k2 = pass_tc_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       IntraSmem<C>::kBytes);
  if (e != cudaSuccess) return e;
  // the whole carveout as shared memory, so that two CTAs fit on an SM
  e = cudaFuncSetAttribute(k1, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, PassSmem<C>::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned pass_ctas = static_cast<unsigned>(p.num_seqs) * a.Hv;

  // Pieces. With few (sequence, value head) pairs the state pass holds few SMs for its whole
  // chain, so the chunks run in pieces, in one stream: intra(0), pass(0), intra(1), pass(1), ...
  // Each later kernel is a programmatic dependent of the one before: intra(k + 1) starts once
  // every CTA of pass(k) is resident (a pass CTA needs an SM of its own: its shared and tensor
  // memory exclude an intra CTA) and runs on the other SMs beside it; its CTA 0 then waits for
  // pass(k) before it exits, so pass(k + 1), which waits for intra(k + 1), finds the state
  // pass(k) left. The first piece is short, so that the first pass starts early, and each next
  // one half as long again: its intra kernel, on the SMs the pass leaves, keeps ahead of the
  // pass before it. The mixed step records its event (before_pass) before the last pass, the
  // longest, beside which no intra kernel runs: its decode rows take the SMs that pass leaves.
  // intra(0) is a programmatic dependent too, of the kernel before it (the chunk table's, or the
  // conv's), and waits for it at entry: its launch overlaps that kernel.
  int bounds[16] = {0, M}, pieces = 1;
  if (static_cast<int64_t>(p.num_seqs) * a.Hv <= kPieceSeqHeads && M >= 16) {
    int n = (max(4, M / 8) + CPC - 1) / CPC * CPC, g = 0;
    pieces = 0;
    while (g < M && pieces < 15) {
      const int left = M - g;
      const int take = (pieces == 14 || left < n + n / 2) ? left : n;  // a short tail joins
      bounds[pieces] = g;
      g += take;
      ++pieces;
      n = (n * 3 / 2 + CPC - 1) / CPC * CPC;
    }
    bounds[pieces] = M;
  }
  float* sx = pieces > 1 ? reinterpret_cast<float*>(ws + L.sx) : nullptr;
  for (int k = 0; k < pieces; ++k) {
    const int g_lo = bounds[k], g_hi = k + 1 < pieces ? bounds[k + 1] : INT_MAX;
    const int n_chunks = bounds[k + 1] - g_lo;
    if (n_chunks > 0) {
      // the first intra kernel of several pieces holds up the first pass: when its CTAs split
      // by value head still fit one wave (two per SM), each takes one head
      const unsigned nx = static_cast<unsigned>((n_chunks + CPC - 1) / CPC);
      const int R = a.Hv / a.Hk;
      const int hsplit = (k == 0 && pieces > 1 && R > 1 &&
                          static_cast<int64_t>(nx) * a.Hk * R <= 2 * static_cast<int64_t>(sm_count()))
                             ? 1 : 0;
      e = launch_k(k1, dim3(nx, a.Hk, hsplit ? R : 1), kThreadsTc, IntraSmem<C>::kBytes, s, true, a,
                   p, y, meta, chunk_off, chunk_seq, wb, g_lo / CPC, k > 0 ? 1 : 0, hsplit,
                   k == 0 ? 1 : 0);
      if (e != cudaSuccess) return e;
    }
    if (k == pieces - 1 && p.before_pass && (e = cudaEventRecord(p.before_pass, s)) != cudaSuccess)
      return e;
    e = launch_k(k2, dim3(pass_ctas), kPassThreads, PassSmem<C>::kBytes, s, pieces > 1, a, p,
                 seq_ok, chunk_off, seq_order, wb, g_lo, g_hi, sx, pieces > 1 ? 1 : 0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t set_prefill_test_fault(int mode) {
  return cudaMemcpyToSymbol(g_test_fault, &mode, sizeof(int));
}

size_t prefill_tc_workspace_bytes(int total_tokens, int num_seqs, int Hk, int Hv, int chunk) {
  return tc_layout(total_tokens, num_seqs, Hk, Hv, chunk, 2 * Hk * kD + Hv * kD).total;
}

cudaError_t launch_prefill_tc(const LayerArgs& a, const PrefillExtra& p, cudaStream_t s) {
  const TcLayout L = tc_layout(p.total_tokens, p.num_seqs, a.Hk, a.Hv, p.chunk, a.D);
  char* ws = static_cast<char*>(p.workspace);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + L.meta);
  int32_t* seq_ok = reinterpret_cast<int32_t*>(ws + L.seq_ok);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_off);
  int32_t* chunk_seq = reinterpret_cast<int32_t*>(ws + L.chunk_seq);
  int32_t* seq_order = reinterpret_cast<int32_t*>(ws + L.seq_order);
  cudaError_t e = launch_prefill_prep(a, p, meta, seq_ok, chunk_off, chunk_seq, seq_order, s);
  if (e != cudaSuccess) return e;
  const uint16_t* y = static_cast<const uint16_t*>(a.mixed);
  if (a.conv_w) {
    uint16_t* ybuf = reinterpret_cast<uint16_t*>(ws + L.ybuf);
    e = launch_prefill_conv(a, p, meta, seq_ok, chunk_off, chunk_seq, L.max_chunks, ybuf, s);
    if (e != cudaSuccess) return e;
    y = ybuf;
  }
  switch (p.chunk) {
    case 16: return launch_tc_c<16>(a, p, L, ws, y, s);
    case 32: return launch_tc_c<32>(a, p, L, ws, y, s);
    case 64: return launch_tc_c<64>(a, p, L, ws, y, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
