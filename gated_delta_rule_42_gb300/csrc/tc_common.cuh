// Shared pieces of the bf16 tensor-core KDA kernels (K, V = 64 or 128 in 128-wide tiles, chunk 64):
// the asynchronous loads and bulk copies, the phase-timing hooks and the
// operand-descriptor helpers.
//
// Every operand tile is 128-byte swizzled (see umma.cuh), so the same bytes
// serve as a K-major or an MN-major tcgen05 operand and as an ldmatrix source.
#pragma once

#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {
namespace tc {

using namespace umma;

// Phase timing (compile with -DKDA_PHASE_TIMING): thread 0 of every block
// adds the clock64 cycles since its previous stamp to a shared-memory slot i
// (KDA_PT(i)); KDA_PT_FLUSH adds the slots to kda_phase_cycles (one copy per
// translation unit, read back by the KDA_PT_EXPORT function), so the totals
// are sums over all blocks.  Off by default; it skips no work.
#ifdef KDA_PHASE_TIMING
static __device__ long long kda_phase_cycles[32];
static __shared__ long long kda_pt_acc[33];  // [32] = time of the last stamp
#ifndef KDA_PT_TID
#define KDA_PT_TID 0  // the thread whose timeline is recorded
#endif
#define KDA_PT_ON (threadIdx.x == KDA_PT_TID)
#define KDA_PT_DECL                                             \
  do {                                                          \
    if (KDA_PT_ON) {                                            \
      for (int i_ = 0; i_ < 32; ++i_) kda_pt_acc[i_] = 0;       \
      kda_pt_acc[32] = clock64();                               \
    }                                                           \
  } while (0)
#define KDA_PT(i)                                   \
  do {                                              \
    if (KDA_PT_ON) {                                \
      const long long now_ = clock64();             \
      kda_pt_acc[i] += now_ - kda_pt_acc[32];       \
      kda_pt_acc[32] = now_;                        \
    }                                               \
  } while (0)
#define KDA_PT_FLUSH                                                            \
  do {                                                                          \
    if (KDA_PT_ON)                                                              \
      for (int i_ = 0; i_ < 32; ++i_)                                           \
        atomicAdd((unsigned long long *)&kda_phase_cycles[i_], (unsigned long long)kda_pt_acc[i_]); \
  } while (0)
#define KDA_PT_EXPORT(name)                                                                      \
  extern "C" int name(long long *out, int reset) {                                               \
    if (cudaMemcpyFromSymbol(out, tc::kda_phase_cycles, sizeof(long long) * 32) != cudaSuccess) \
      return 1;                                                                                  \
    static const long long z[32] = {};                                                           \
    if (reset && cudaMemcpyToSymbol(tc::kda_phase_cycles, z, sizeof(z)) != cudaSuccess) return 1; \
    return 0;                                                                                    \
  }
#else
#define KDA_PT_DECL \
  do {              \
  } while (0)
#define KDA_PT(i) \
  do {            \
  } while (0)
#define KDA_PT_FLUSH \
  do {               \
  } while (0)
#define KDA_PT_EXPORT(name)
#endif

constexpr int kC = 64;     // chunk
constexpr int kD = 128;    // the tiles' K = V (a 64-wide head is zero-padded to it)
constexpr int kThr = 256;  // 8 warps
constexpr int kGLD = 132;  // padded fp32 row stride of the gate tile of the per-chunk gradient kernel
constexpr int kGT = 128;   // row stride of the TMA-loaded gate tile (dense rows)

// The KDA gate over a chunk's [64][ld] gate tile in shared memory (raw
// pre-activations in, the per-token log2 decay out), elementwise over NT
// threads (t: the calling thread's index among them): rows < len, channels < K
// (the rest is never summed).
template <int NT>
__device__ __forceinline__ void kgate_tile(float *G, int ld, int len, int K, int j, const GateArgs &ga, int t) {
  static_assert(NT % 128 == 0, "each thread keeps one channel");
  const int c = t & 127;
  if (c >= K) return;
  const float sc = kgate_scale(ga, j), b = kgate_bias(ga, K, j, c);
  if (NT >= 512) {  // few rows per thread: all of them at once
#pragma unroll
    for (int i = 0; i < kC / (NT / 128); ++i) {
      const int r = (t >> 7) + i * (NT / 128);
      if (r < len) G[r * ld + c] = kgate_fast(G[r * ld + c] + b, sc, ga.lb);
    }
  } else {
    for (int r = t >> 7; r < len; r += NT / 128) G[r * ld + c] = kgate_fast(G[r * ld + c] + b, sc, ga.lb);
  }
}
// The same over the whole CTA (NT threads).
template <int NT = kThr>
__device__ __forceinline__ void kgate_tile(float *G, int ld, int len, int K, int j, const GateArgs &ga) {
  kgate_tile<NT>(G, ld, len, K, j, ga, (int)threadIdx.x);
}

// 1 / sqrt(K) for the head dims of the tensor-core path (64 or 128), exactly.
__host__ __device__ __forceinline__ float head_qscale(int K) { return K == 64 ? 0.125f : 0.08838834764831845f; }

// rows of the per-channel vector table of the per-chunk gradient kernel: G_last,
// 2^G_last, the row references Gr(R) and 2^Gr(R), the block-pair factors D_RI,
// 2^(G_last - Gc(R)) and the column references Gc(R)
constexpr int V_GL = 0, V_GAML = 1, V_RREF = 2, V_EREF = 6, V_D = 10, V_LAM = 16, V_CREF = 20;

__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void st_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};\n" ::"r"(dst), "r"(0u) : "memory");
}
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                    pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ void unpack8(uint4 u, float (&x)[8]) {
  float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), c = unpack_bf16(u.z), d = unpack_bf16(u.w);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}

// Descriptor of 16-row K slice s of an MN-major operand stored as a swizzled
// tile whose rows are the K index (row stride 128 B) and whose columns are the
// M (or N) index in 64-wide sub-tiles `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int s, uint32_t lbo) {
  uint64_t d = (uint64_t)(((tile + (uint32_t)s * 2048u) >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16 instruction descriptor with operand majors (0 = K-major, 1 = MN-major).
__device__ __forceinline__ uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return idesc_bf16(M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}

// 2^x for the per-element decay factors: one hardware base-2 exponential (PTX
// ex2.approx.ftz.f32, within about 2 ulp; results below 2^-126 flush to zero).
// The block factors it serves lie within 2^-96 .. 2^96, or are <= 1.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Asynchronous loads of one chunk's gate rows ([tokens][HV][K] fp32, K = 64 or
// 128) into a [64][kGLD] tile; rows at or past len and channels past K are zeroed.
template <int NT = kThr>
__device__ __forceinline__ void load_gate(uint32_t tile, const float *g, int t0, int len, int HV, int j, int K) {
  for (int it = threadIdx.x; it < kC * 32; it += NT) {
    const int r = it >> 5, jj = it & 31;
    const uint32_t dst = tile + (uint32_t)(r * kGLD + jj * 4) * 4u;
    if (r < len && jj * 4 < K) cp16(dst, g + ((size_t)(t0 + r) * HV + j) * K + jj * 4);
    else st_zero16(dst);
  }
}

// First token and length of chunk ci of a sequence whose table entry is
// si = (first token, length, first chunk, chunk count): computed, not loaded,
// so the sequential kernels never wait on the chunk table.
__device__ __forceinline__ int2 chunk_span(const int4 &si, int ci) {
  const int t = kC * ci;
  return make_int2(si.x + t, min(kC, si.y - t));
}

// ---- TMA (bulk tensor) loads of the per-token tiles ----
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Contiguous global -> shared bulk copy (16-byte aligned, size a multiple of 16); completion on bar.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Contiguous shared -> global bulk copy (16-byte aligned, size a multiple of 16), in the
// calling thread's bulk group; the source must stay unchanged until bulk_wait_read().
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// The calling thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// All but the most recent of the calling thread's bulk store groups have read their sources.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory");
}
// The calling thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
// Box (c0, c1, c2) of a 3-D tensor map into shared memory; completion counted on bar.
__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::
          "r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
// One swizzled [64][128] bf16 tile = two 64 x 64 boxes (channel offsets 0 and 64).
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int head, int t0, uint64_t *bar) {
  tma_load3(dst, map, 0, head, t0, bar);
  tma_load3(dst + 8192, map, 64, head, t0, bar);
}
// Rows len..63 of a swizzled [64][128] bf16 tile -> 0 (after its load completed).
template <int NT = kThr>
__device__ __forceinline__ void zero_tail(unsigned char *tile, int len) {
  for (int it = threadIdx.x; it < (kC - len) * 16; it += NT) {
    const int r = len + (it >> 4), q = it & 15;
    *reinterpret_cast<uint4 *>(tile + (q >> 3) * 8192 + r * 128 + (q & 7) * 16) = make_uint4(0, 0, 0, 0);
  }
}
// beta of one chunk (asynchronous; zero past len).
__device__ __forceinline__ void load_beta(const Problem &P, float *dst, int t0, int len, int j) {
  if (threadIdx.x < kC) {
    if (threadIdx.x < len) cp4(smem_u32(dst + threadIdx.x), P.beta + (size_t)(t0 + threadIdx.x) * P.HV + j);
    else dst[threadIdx.x] = 0.f;
  }
}

}  // namespace tc
}  // namespace kda
