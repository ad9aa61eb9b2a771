// gdn_tc.cuh -- 5th-generation tensor core (tcgen05) helpers for sm_100-class
// GPUs, written as inline PTX: tensor-memory allocation, shared-memory matrix
// descriptors, the instruction descriptor of kind::f16 (bf16 in, fp32
// accumulate), MMA issue / commit, and tensor-memory loads.
//
// Operand layout used throughout (no swizzle, "K-major"): a bf16 tile of R rows
// by K columns is stored as 8x8 core matrices of 128 contiguous bytes (8 rows
// of 16 bytes); the core matrices of one 8-row group follow each other along K
// (leading-dimension byte offset LBO = 128), and 8-row groups are K*16 bytes
// apart (stride-dimension byte offset SBO = K * 16). Element (r, k) therefore
// sits at byte  (r / 8) * K * 16 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
// One MMA consumes K = 16 (two core-matrix columns); the next K step starts
// 256 bytes further on.
//
// Accumulators (M = 128, cta_group::1): row i of D lives in tensor-memory lane
// i, column j in column (base + j); warp w of the CTA may access lanes
// 32 * (w % 4) .. 32 * (w % 4) + 31. An A operand may live in tensor memory too
// (mma_bf16_ts), row m in lane m, two bf16 of K per column.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_ptx.cuh"

namespace gdn {
namespace tc {

// byte offset of bf16 element (r, k) inside a K-major no-swizzle tile
__host__ __device__ __forceinline__ uint32_t kmajor_offset(int r, int k, int K) {
  return static_cast<uint32_t>((r >> 3) * K * 16 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor (sm_100 format, no swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for sm_100
  return d;                             // base offset 0, swizzle none
}

// Descriptor of the K-step `ks` (16 columns) of a K-major tile with K columns.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_saddr, int K, int ks) {
  return smem_desc(tile_saddr + static_cast<uint32_t>(ks) * 256u, 128u, static_cast<uint32_t>(K) * 16u);
}

// Descriptor of the K-step `ks` (16 K-rows) of an MN-major tile [K x N] stored in the K-major
// tile layout with the roles swapped: element (k, n) at kmajor_offset(k, n, N), i.e. core
// matrices of 8 K-rows x 16 bytes of N, 128 bytes apart along N and N*16 bytes apart along K.
// For an MN-major operand (no swizzle) the leading byte offset is the K stride and the
// stride byte offset the N stride (checked against exact integer products before use).
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile_saddr, int N, int ks) {
  return smem_desc(tile_saddr + static_cast<uint32_t>(ks) * 32u * static_cast<uint32_t>(N),
                   static_cast<uint32_t>(N) * 16u, 128u);
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}
// The same with an MN-major B operand (bit 16: B transposed).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_bmn(int M, int N) {
  return idesc_bf16_f32(M, N) | (1u << 16);
}
// The same with an MN-major A operand (bit 15: A transposed); its descriptor takes the same
// strides as an MN-major B (mnmajor_desc with M in place of N).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_amn(int M, int N) {
  return idesc_bf16_f32(M, N) | (1u << 15);
}

// --- tensor memory allocation (executed by one whole warp) ---
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// --- MMA issue (one thread) ---
// D[tmem] (+)= A[smem] * B[smem]^T ; accumulate = 0 overwrites D.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with the A operand in tensor memory (M = 128: row m in lane m; K = 16 per MMA as 8
// columns, each holding the bf16 pair (k, k + 1) with element k in the low half; checked
// against exact integer products before use).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on an mbarrier when every MMA this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy writes to shared memory -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --- tensor memory -> registers: 32 lanes x 16 columns of 32 bits per warp ---
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// --- registers -> tensor memory: 32 lanes x 4 columns of 32 bits per warp (lane = thread) ---
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint4& v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
               "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
               "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
               "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
               "f"(v[15])
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// tensor-memory address of (lane, column)
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane, int col) {
  return base + (static_cast<uint32_t>(lane) << 16) + static_cast<uint32_t>(col);
}

}  // namespace tc
}  // namespace gdn
