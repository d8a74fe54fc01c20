// Blackwell (sm_103a) tensor-core helpers: tcgen05 MMA with operands in
// shared memory (UMMA descriptors), accumulators in tensor memory (TMEM),
// mbarrier completion tracking, and the 128-byte-swizzled K-major tile layout
// every tensor-core operand in this library uses.  Also the legacy warp-level
// mma.sync / ldmatrix wrappers used for the small 16x16 blocks.
//
// Every wait on an mbarrier is bounded: after kSpinLimit polls it gives up and
// raises the caller's error flag instead of hanging the GPU.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {
namespace umma {

constexpr long kSpinLimit = 1L << 24;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- 128B-swizzled K-major tiles -------------------------------------------
// A tile of R rows (R % 8 == 0) and W bf16 columns (W = 64 or 128) is stored as
// W/64 sub-tiles of [R][64] (128 bytes per row), each 1024-byte aligned.  In a
// sub-tile the 16-byte chunk j of row r sits at chunk position j ^ (r % 8):
// the canonical SWIZZLE_128B K-major layout of the UMMA descriptor, and also
// conflict-free for ldmatrix and for 16-byte row accesses.
__device__ __forceinline__ uint32_t sw_off(int r, int c, int R) {
  const int sub = c >> 6, cc = c & 63;
  return (uint32_t)sub * (uint32_t)R * 128u + (uint32_t)r * 128u +
         ((uint32_t)((cc >> 3) ^ (r & 7)) << 4) + (uint32_t)(cc & 7) * 2u;
}
// byte offset of the 16-byte chunk holding columns [8*j, 8*j+8) of row r
__device__ __forceinline__ uint32_t sw_chunk(int r, int j, int R) {
  const int sub = j >> 3, jj = j & 7;
  return (uint32_t)sub * (uint32_t)R * 128u + (uint32_t)r * 128u + ((uint32_t)(jj ^ (r & 7)) << 4);
}

// Shared-memory matrix descriptor for a SWIZZLE_128B K-major operand whose
// 8-row core groups are 1024 bytes apart.  `addr` is the shared address of the
// first element of the 16-column K slice (sub-tile base + 32 * (k16 % 4)).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;            // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;            // SWIZZLE_128B
  return d;
}
// Descriptor of K slice k16 (16 columns) of a tile of R rows.
__device__ __forceinline__ uint64_t desc_k16(uint32_t tile, int k16, int R) {
  return desc_sw128(tile + (uint32_t)(k16 >> 2) * (uint32_t)R * 128u + (uint32_t)(k16 & 3) * 32u);
}

// Instruction descriptor: kind::f16, bf16 A and B, fp32 accumulator, both
// operands K-major, M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T with A: M x 16 and B: N x 16 (K-major descriptors).
__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive on `bar` once every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void bar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and sets *err) after `limit` unsuccessful polls.
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity, int *err, long limit = kSpinLimit) {
  for (long it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  if (err) atomicExch(err, 1);
  return false;
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// TMEM allocation (one full warp executes these).
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(slot)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}

// 16 (tmem_ld16) or 32 (tmem_ld32) consecutive fp32 columns of this thread's
// TMEM lane (warp-collective).  The warp must address its own lane quarter:
// lane base 32 * (warp % 4).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Three 16-lane x 8-column blocks of fp32 accumulators (lane base: the warp's
// quarter, + column offsets a0, a1, a2) in mma.sync C-fragment order: thread t
// gets (lane t/4, columns 2(t%4), 2(t%4)+1) then (lane t/4 + 8, the same columns).
__device__ __forceinline__ void tmem_ld_frag3(uint32_t a0, uint32_t a1, uint32_t a2, float (&x)[4], float (&y)[4],
                                              float (&z)[4]) {
  uint32_t r[12];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%12];\n"
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%4,%5,%6,%7}, [%13];\n"
      "tcgen05.ld.sync.aligned.16x256b.x1.b32 {%8,%9,%10,%11}, [%14];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11])
      : "r"(a0), "r"(a1), "r"(a2)
      : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[i] = __uint_as_float(r[i]);
    y[i] = __uint_as_float(r[4 + i]);
    z[i] = __uint_as_float(r[8 + i]);
  }
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- legacy warp MMA (16x8x16 bf16, fp32 accumulate) -------------------------
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&t);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 t = *reinterpret_cast<__nv_bfloat162 *>(&u);
  return __bfloat1622float2(t);
}

}  // namespace umma
}  // namespace kda
