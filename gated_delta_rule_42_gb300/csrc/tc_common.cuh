// Shared pieces of the fused bf16 tensor-core KDA kernels (K = V = 128,
// chunk 64): the shared-memory map, the asynchronous chunk loads, and the two
// V-independent phases every chunk step needs:
//  (a) chunk-local cumsum G of the log2 gate and the decay-scaled operand tiles;
//  (b) the decayed Gram blocks L (strictly lower, beta-scaled) and Aqk (lower)
//      on 16x16 warp MMAs, and A = (I + L)^-1 in fp32.
//
// Decay scaling.  2^(G_r - G_i) is split at the first row of each 16-token
// block (ref): rows carry 2^(G_r - G_ref) <= 1 (tile Kr / Qr), columns carry
// 2^(G_ref - G_i) <= 2^(15 |g|max) (tile Kc), and between blocks the per-channel
// factor D_RI = 2^(G_ref(R) - G_ref(I)) <= 1 is applied to the column fragments
// in registers.  Nothing overflows for gates >= -8 per token (log2 units).  The
// chunk-level tiles Bk = beta k 2^G, Qg = q~ 2^G and Khat = k 2^(G_last - G)
// only underflow where the true value is negligible.
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
#define KDA_PT_ON (threadIdx.x == 0)
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
constexpr int kD = 128;    // K = V
constexpr int kThr = 256;  // 8 warps
constexpr int kGLD = 132;  // padded fp32 row stride of the gate tile of the chain kernel
constexpr int kGT = 128;   // row stride of the TMA-loaded gate tile of the sequential kernels

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KRAW = 0;       // k  [64][128] bf16
constexpr uint32_t OFF_QRAW = 16384;   // q  [64][128]
constexpr uint32_t OFF_VRAW = 32768;   // v (forward) or dO (backward) [64][128]
constexpr uint32_t OFF_GRAW = 49152;   // g -> G  fp32 [64][128] (dense rows: a TMA box)
constexpr uint32_t OFF_BK = 83968;     // beta k 2^G         [64 r][128 c]
constexpr uint32_t OFF_QG = 100352;    // q~ 2^G             [64 r][128 c]
constexpr uint32_t OFF_KH = 116736;    // k 2^(G_last - G)   [64 r][128 c]
constexpr uint32_t OFF_AQK = 133120;   // Aqk                [64 r][64 i]
constexpr uint32_t OFF_AM = 141312;    // A = (I + L)^-1     [64 r][64 i]
constexpr uint32_t OFF_U = 149504;     // union (64 KB): phases (a)/(b) | phase (c)
constexpr uint32_t U_KR = 0, U_QR = 16384, U_KC = 32768, U_LF = 49152;  // (a)/(b)
constexpr uint32_t U_AF = 0, U_T = 16384;                              // (b) inverse scratch
constexpr uint32_t OFF_VEC = 215040;   // fp32 vectors (20 rows of 128)
constexpr uint32_t OFF_BETA = 225280;  // beta, two buffers of 64 fp32
constexpr uint32_t OFF_MISC = 225792;  // mbarriers (MMA +0, k/q/g loads +16, v loads +24, output MMA +32), tmem slot +8
constexpr uint32_t SMEM_BYTES = 225792 + 64 + 1024;  // + alignment slack
constexpr int V_GL = 0, V_GAML = 1, V_GREF = 2, V_EREF = 6, V_D = 10, V_LAM = 16;
static_assert(OFF_QG == OFF_BK + 16384 && OFF_KH == OFF_QG + 16384 && OFF_AQK == OFF_KH + 16384 &&
                  OFF_AM == OFF_AQK + 8192 && OFF_AM - OFF_BK == kTileRecA && OFF_AM + 8192 - OFF_BK == 65536,
              "the saved tile record is the contiguous Bk .. A region");

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
__device__ __forceinline__ void st_bf2(unsigned char *tile, int r, int c, int R, float a, float b) {
  *reinterpret_cast<uint32_t *>(tile + sw_off(r, c, R)) = pack_bf16(a, b);
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

// Asynchronous loads of one chunk's rows of a [tokens][heads][128] bf16
// tensor into a swizzled [64][128] tile; rows at or past len are zeroed.
template <int NT = kThr>
__device__ __forceinline__ void load_rows(uint32_t tile, const __nv_bfloat16 *src, int t0, int len,
                                          int heads, int head) {
  for (int it = threadIdx.x; it < kC * 16; it += NT) {
    const int r = it >> 4, jj = it & 15;
    const uint32_t dst = tile + sw_chunk(r, jj, kC);
    if (r < len) cp16(dst, src + ((size_t)(t0 + r) * heads + head) * kD + jj * 8);
    else st_zero16(dst);
  }
}

template <int NT = kThr>
__device__ __forceinline__ void load_gate(uint32_t tile, const float *g, int t0, int len, int HV, int j) {
  for (int it = threadIdx.x; it < kC * 32; it += NT) {
    const int r = it >> 5, jj = it & 31;
    const uint32_t dst = tile + (uint32_t)(r * kGLD + jj * 4) * 4u;
    if (r < len) cp16(dst, g + ((size_t)(t0 + r) * HV + j) * kD + jj * 4);
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
// k, q (when with_q) and the gate rows of one chunk, issued by one thread:
// rows past the tensor end arrive as zeros, rows past the sequence end hold
// the next tokens (zero_tail clears them where it matters).
__device__ __forceinline__ void tma_kqg(const TmaMaps &M, uint32_t base, int t0, int h, int j, bool with_q,
                                        uint64_t *bar) {
  mbar_expect_tx(bar, (with_q ? 32768u : 16384u) + 32768u);
  tma_tile(base + OFF_KRAW, &M.k, h, t0, bar);
  if (with_q) tma_tile(base + OFF_QRAW, &M.q, h, t0, bar);
  tma_load3(base + OFF_GRAW, &M.g, 0, j, t0, bar);
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

// Phase (a).  Needs the k (and q) staging tiles, the gate tile and beta of the
// chunk; ends with a __syncthreads.  Writes G (in place), the vectors, and the
// tiles Bk, Khat (and Qg when kQ); with kGram also the decay tiles Kr, Kc (and
// Qr) that the Gram blocks of phase (b) need.
template <bool kQ, bool kGram = true>
__device__ __forceinline__ void phase_a(unsigned char *sm, int len, const float *beta) {
  const int tid = threadIdx.x;
  float *G = (float *)(sm + OFF_GRAW);
  float *vec = (float *)(sm + OFF_VEC);
  unsigned char *U = sm + OFF_U;
  constexpr float qscale = 0.08838834764831845f;  // 1/sqrt(128)
  {  // two threads per channel (adjacent lanes), 32 rows each
    const int c = tid >> 1, hf = tid & 1, r0 = 32 * hf, lane = tid & 31;
    float col[32];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) col[k] = G[(r0 + k) * kGT + c];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      if (r0 + k < len) s += col[k];
      col[k] = s;
    }
    const float lo_total = __shfl_sync(0xffffffffu, s, lane & ~1);
    const float add = hf ? lo_total : 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      col[k] += add;
      G[(r0 + k) * kGT + c] = col[k];
    }
    const float gl = __shfl_sync(0xffffffffu, s + add, lane | 1);
    // block references: rows 0, 16 (lower partner) and 32, 48 (upper partner)
    const float ga = (r0 < len) ? col[0] : gl, gb = (r0 + 16 < len) ? col[16] : gl;
    float gref[4];
    gref[0] = __shfl_sync(0xffffffffu, ga, lane & ~1);
    gref[1] = __shfl_sync(0xffffffffu, gb, lane & ~1);
    gref[2] = __shfl_sync(0xffffffffu, ga, lane | 1);
    gref[3] = __shfl_sync(0xffffffffu, gb, lane | 1);
    if (hf == 0) {
      vec[V_GL * kD + c] = gl;
      vec[V_GAML * kD + c] = exp2f(gl);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // this partner's own two references (ga, gb)
      const int R = 2 * hf + q;
      const float gr = q ? gb : ga;
      vec[(V_GREF + R) * kD + c] = gr;
      vec[(V_EREF + R) * kD + c] = exp2f(gr);
      vec[(V_LAM + R) * kD + c] = exp2f(gl - gr);
    }
    // D_RI = 2^(gref_R - gref_I) for the pairs (1,0) (2,0) (2,1) | (3,0) (3,1) (3,2)
    if (hf == 0) {
      vec[(V_D + 0) * kD + c] = exp2f(gref[1] - gref[0]);
      vec[(V_D + 1) * kD + c] = exp2f(gref[2] - gref[0]);
      vec[(V_D + 2) * kD + c] = exp2f(gref[2] - gref[1]);
    } else {
      vec[(V_D + 3) * kD + c] = exp2f(gref[3] - gref[0]);
      vec[(V_D + 4) * kD + c] = exp2f(gref[3] - gref[1]);
      vec[(V_D + 5) * kD + c] = exp2f(gref[3] - gref[2]);
    }
  }
  __syncthreads();
  KDA_PT(1);
  // thread: 8 consecutive channels (one 16-byte chunk) of 4 consecutive rows
  {
    const int jj = tid & 15, c0 = jj * 8, rg = tid >> 4, R = rg >> 2;
    float gref[8], eref[8], lam[8];
#pragma unroll
    for (int e = 0; e < 8; e += 4) {
      *reinterpret_cast<float4 *>(gref + e) = *reinterpret_cast<const float4 *>(vec + (V_GREF + R) * kD + c0 + e);
      *reinterpret_cast<float4 *>(eref + e) = *reinterpret_cast<const float4 *>(vec + (V_EREF + R) * kD + c0 + e);
      *reinterpret_cast<float4 *>(lam + e) = *reinterpret_cast<const float4 *>(vec + (V_LAM + R) * kD + c0 + e);
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = rg * 4 + rr;
      const uint32_t off = sw_chunk(r, jj, kC);
      float kv[8], qv[8], g[8], e1[8], e2[8], o[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_KRAW + off), kv);
      if (kQ) unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_QRAW + off), qv);
      *reinterpret_cast<float4 *>(g) = *reinterpret_cast<const float4 *>(G + r * kGT + c0);
      *reinterpret_cast<float4 *>(g + 4) = *reinterpret_cast<const float4 *>(G + r * kGT + c0 + 4);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        e1[e] = exp2f(g[e] - gref[e]);  // <= 1
        e2[e] = exp2f(gref[e] - g[e]);  // >= 1
      }
      const float br = beta[r];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e1[e];
      if (kGram) *reinterpret_cast<uint4 *>(U + U_KR + off) = pack8(o);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e];
      if (kGram) *reinterpret_cast<uint4 *>(U + U_KC + off) = pack8(o);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = br * kv[e] * e1[e] * eref[e];
      *reinterpret_cast<uint4 *>(sm + OFF_BK + off) = pack8(o);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e] * lam[e];
      *reinterpret_cast<uint4 *>(sm + OFF_KH + off) = pack8(o);
      if (kQ) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = qv[e] * qscale * e1[e];
        if (kGram) *reinterpret_cast<uint4 *>(U + U_QR + off) = pack8(o);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= eref[e];
        *reinterpret_cast<uint4 *>(sm + OFF_QG + off) = pack8(o);
      }
    }
  }
  __syncthreads();
}

// fp32 [64][64] scratch of phase (b) (L, then A): columns XOR-swizzled by
// 4 * (row % 8), so reads of one column across 8 rows and float4 reads of four
// consecutive columns are both free of bank conflicts.
__device__ __forceinline__ int fsw(int r, int c) { return r * kC + (c ^ ((r & 7) << 2)); }

// Phase (b).  Needs the tiles of phase (a); ends with a __syncthreads.  Writes
// the A tile (and the Aqk tile when kQ).  Clobbers the union region.
template <bool kQ>
__device__ __forceinline__ void phase_b(unsigned char *sm, const float *beta) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(sm);
  const float *vec = (const float *)(sm + OFF_VEC);
  unsigned char *U = sm + OFF_U;
  float *Lf = (float *)(U + U_LF);
  // Gram blocks: the 10 block pairs R >= I over the 8 warps (the A fragments of
  // a pair serve both 8-column halves: shared-memory wavefronts bound this phase).
  for (int p = warp; p < 10; p += 8) {
    const int R = p >= 6 ? 3 : p >= 3 ? 2 : p >= 1 ? 1 : 0, I = p - R * (R + 1) / 2;
    const float *Dv = (I < R) ? vec + (V_D + R * (R - 1) / 2 + I) * kD : nullptr;
    float accL[2][4] = {}, accQ[2][4] = {};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t ak[4], aq[4] = {0, 0, 0, 0}, b[4];
      {
        const int row = 16 * R + (lane & 7) + ((lane >> 3) & 1) * 8, jj = 2 * s + (lane >> 4);
        ldsm_x4(sbase + OFF_U + U_KR + sw_chunk(row, jj, kC), ak[0], ak[1], ak[2], ak[3]);
        if (kQ) ldsm_x4(sbase + OFF_U + U_QR + sw_chunk(row, jj, kC), aq[0], aq[1], aq[2], aq[3]);
      }
      {
        const int mi = lane >> 3;
        const int row = 16 * I + (lane & 7) + (mi >> 1) * 8, jj = 2 * s + (mi & 1);
        ldsm_x4(sbase + OFF_U + U_KC + sw_chunk(row, jj, kC), b[0], b[1], b[2], b[3]);
      }
      if (Dv != nullptr) {
        const int c0 = 16 * s + (lane & 3) * 2;
        const float2 d01 = *reinterpret_cast<const float2 *>(Dv + c0);
        const float2 d89 = *reinterpret_cast<const float2 *>(Dv + c0 + 8);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = unpack_bf16(b[t]);
          b[t] = (t & 1) ? pack_bf16(f.x * d89.x, f.y * d89.y) : pack_bf16(f.x * d01.x, f.y * d01.y);
        }
      }
      mma16816(accL[0], ak, b[0], b[1]);
      mma16816(accL[1], ak, b[2], b[3]);
      if (kQ) {
        mma16816(accQ[0], aq, b[0], b[1]);
        mma16816(accQ[1], aq, b[2], b[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * R + (lane >> 2) + hh * 8;
        const int i = 16 * I + nt * 8 + (lane & 3) * 2;
        const float br = beta[r];
        const float l0 = (i < r) ? br * accL[nt][2 * hh] : 0.f;
        const float l1 = (i + 1 < r) ? br * accL[nt][2 * hh + 1] : 0.f;
        *reinterpret_cast<float2 *>(Lf + fsw(r, i)) = make_float2(l0, l1);
        if (kQ) {
          const float a0 = (i <= r) ? accQ[nt][2 * hh] : 0.f;
          const float a1 = (i + 1 <= r) ? accQ[nt][2 * hh + 1] : 0.f;
          st_bf2(sm + OFF_AQK, r, i, kC, a0, a1);
        }
      }
    }
  }
  if (kQ && tid < 6 * 32) {  // Aqk blocks above the diagonal (R < I) are zero
    const int b = tid >> 5, w = tid & 31;
    const int R = (b < 3) ? 0 : (b < 5 ? 1 : 2), I = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
    *reinterpret_cast<uint4 *>(sm + OFF_AQK + sw_chunk(16 * R + (w >> 1), 2 * I + (w & 1), kC)) = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  KDA_PT(4);
  float *Af = (float *)(U + U_AF);  // overwrites Kr (dead)
  float *Tf = (float *)(U + U_T);   // overwrites Qr (dead)
  if (warp < 4 && lane < 16) {
    // diagonal block R = warp: lane i computes column i of (I + L_RR)^-1
    const int R = warp, i = lane;
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) a[m] = (m == i) ? 1.f : 0.f;
    // column-oriented substitution: once a[m] is final, subtract its multiples
    // from every later row (independent updates: a short dependency chain);
    // L is read four columns at a time (one float4 per row and column group)
#pragma unroll
    for (int mg = 0; mg < 4; ++mg) {
      float4 lr[16];
#pragma unroll
      for (int r = 4 * mg + 1; r < 16; ++r)
        lr[r] = *reinterpret_cast<const float4 *>(Lf + fsw(16 * R + r, 16 * R + 4 * mg));
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const int m = 4 * mg + mm;
#pragma unroll
        for (int r = m + 1; r < 16; ++r) {
          const float l = mm == 0 ? lr[r].x : mm == 1 ? lr[r].y : mm == 2 ? lr[r].z : lr[r].w;
          a[r] = fmaf(-l, a[m], a[r]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) Af[fsw(16 * R + m, 16 * R + i)] = a[m];
  }
  for (int e = tid; e < 6 * 256; e += kThr) {  // strictly-upper blocks of A
    const int b = e >> 8, w = e & 255;
    const int R = (b < 3) ? 0 : (b < 5 ? 1 : 2);
    const int I = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
    Af[fsw(16 * R + (w >> 4), 16 * I + (w & 15))] = 0.f;
  }
  __syncthreads();
  KDA_PT(5);
  // Off-diagonal blocks, 32-blocked: A = [[A1, 0], [A21, A2]] with A21 = -A2 L21 A1,
  // where A1 = [[D0, 0], [-D1 L10 D0, D1]] and A2 likewise from D2, D3 (D_R the
  // diagonal-block inverses above).  Each thread forms 1 x 4 row segments.
  for (int e = tid; e < 2 * 64; e += kThr) {  // T_b = L_{R,R-1} D_{R-1} for R = 1, 3
    const int b = e >> 6, R = 2 * b + 1, rr = (e >> 2) & 15, i4 = (e & 3) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float l = Lf[fsw(16 * R + rr, 16 * (R - 1) + m)];
      const float4 a = *reinterpret_cast<const float4 *>(Af + fsw(16 * (R - 1) + m, 16 * (R - 1) + i4));
      acc.x = fmaf(l, a.x, acc.x); acc.y = fmaf(l, a.y, acc.y);
      acc.z = fmaf(l, a.z, acc.z); acc.w = fmaf(l, a.w, acc.w);
    }
    *reinterpret_cast<float4 *>(Tf + (b * 16 + rr) * 16 + i4) = acc;
  }
  __syncthreads();
  KDA_PT(16);
  for (int e = tid; e < 2 * 64; e += kThr) {  // A_{R,R-1} = -D_R T_b
    const int b = e >> 6, R = 2 * b + 1, rr = (e >> 2) & 15, i4 = (e & 3) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float l = Af[fsw(16 * R + rr, 16 * R + m)];
      const float4 t = *reinterpret_cast<const float4 *>(Tf + (b * 16 + m) * 16 + i4);
      acc.x = fmaf(l, t.x, acc.x); acc.y = fmaf(l, t.y, acc.y);
      acc.z = fmaf(l, t.z, acc.z); acc.w = fmaf(l, t.w, acc.w);
    }
    *reinterpret_cast<float4 *>(Af + fsw(16 * R + rr, 16 * (R - 1) + i4)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncthreads();
  KDA_PT(17);
  if (tid < 128) {  // 32 x 32 products as 2 x 4 register tiles (rows rg, rg + 16) on four warps
    const int rg = tid >> 3, c4 = (tid & 7) * 4;
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {  // T2 = L21 A1  (A1 lower triangular: zeros above)
      const float4 a = *reinterpret_cast<const float4 *>(Af + fsw(m, c4));
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float l = Lf[fsw(32 + rg + 16 * k, m)];
        acc[k].x = fmaf(l, a.x, acc[k].x); acc[k].y = fmaf(l, a.y, acc[k].y);
        acc[k].z = fmaf(l, a.z, acc[k].z); acc[k].w = fmaf(l, a.w, acc[k].w);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) *reinterpret_cast<float4 *>(Tf + (rg + 16 * k) * 32 + c4) = acc[k];
  }
  __syncthreads();
  KDA_PT(18);
  if (tid < 128) {
    const int rg = tid >> 3, c4 = (tid & 7) * 4;
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {  // A21 = -A2 T2
      const float4 t = *reinterpret_cast<const float4 *>(Tf + m * 32 + c4);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float l = Af[fsw(32 + rg + 16 * k, 32 + m)];
        acc[k].x = fmaf(l, t.x, acc[k].x); acc[k].y = fmaf(l, t.y, acc[k].y);
        acc[k].z = fmaf(l, t.z, acc[k].z); acc[k].w = fmaf(l, t.w, acc[k].w);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k)
      *reinterpret_cast<float4 *>(Af + fsw(32 + rg + 16 * k, c4)) = make_float4(-acc[k].x, -acc[k].y, -acc[k].z, -acc[k].w);
  }
  __syncthreads();
  KDA_PT(19);
  for (int e = tid; e < kC * kC / 8; e += kThr) {  // A -> bf16 tile, 16-byte chunks
    const int r = e >> 3, jj = e & 7;
    float x[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) x[t] = Af[fsw(r, jj * 8 + t)];
    *reinterpret_cast<uint4 *>(sm + OFF_AM + sw_chunk(r, jj, kC)) = pack8(x);
  }
  fence_async_smem();  // the tiles may be read next by the async proxy (bulk stores)
  __syncthreads();
  KDA_PT(6);
}

}  // namespace tc
}  // namespace kda
