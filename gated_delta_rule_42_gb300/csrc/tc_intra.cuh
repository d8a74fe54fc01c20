// Pieces shared by the two per-chunk gradient kernels of the bf16 backward
// (the chunk-reference kernel and the 16-token block-reference kernel): the
// shared-memory map of their input and chain tiles, the slot walk, the three
// groups of input copies and the warp-MMA fragment helpers.
#pragma once

#include "tc_common.cuh"

namespace kda {
namespace intra {

using namespace umma;
using namespace tc;

// Shared memory map (bytes from a 1024-aligned base).  [0, 160 KB) first holds
// the operands of the tensor-core products, then the chain tiles.  "hi/lo"
// tiles hold a value as the sum of two bf16 numbers, so products over
// hi*hi + hi*lo + lo*hi keep ~16 mantissa bits: the pairwise decay terms of
// the chain sum to zero over a chunk and dg accumulates them, so their
// rounding must stay far below the bf16 level.
constexpr uint32_t I_XT = 0;          // X^T [128 v][64 r]  (saved by the forward recompute)
constexpr uint32_t I_DT = 16384;      // D^T [128 v][64 r]  (adjacent: [X; D]^T is one MN-major operand)
constexpr uint32_t I_STK = 32768;     // [dX; dO; dD] [192][128]
constexpr uint32_t I_H = 81920;       // h  [128 c][128 v]
constexpr uint32_t I_DH = 114688;     // dh' [128 c][128 v]
constexpr uint32_t I_V = 147456;      // v  [64 r][128 v]
constexpr uint32_t C_KR = 0;          // Kr  hi [64][128] | lo (+16 KB)
constexpr uint32_t C_QR = 32768;      // Qr  hi | lo
constexpr uint32_t C_KC = 65536;      // Kc  hi | lo
constexpr uint32_t C_DAB = 98304;     // dA^T [64 i][64 m] hi | lo (+8 KB) -> later dL [64 r][64 i] hi | lo
constexpr uint32_t C_DQK = 114688;    // dAqk^T [64 i][64 r] hi | lo
constexpr uint32_t C_XB = 131072;     // X = beta dL [64 r][64 i] hi | lo   (before: raw k rows)
constexpr uint32_t C_T = 147456;      // T = A^T dA [64 r][64 m] hi | lo    (before: raw q rows)
constexpr uint32_t C_KRAW = C_XB, C_QRAW = C_T;
constexpr uint32_t C_G = 163840;      // G fp32 [64][132]
constexpr uint32_t C_A = 197632;      // A   [64 r][64 i] bf16
constexpr uint32_t C_VEC = 205824;    // vectors (24 x 128 fp32)
constexpr uint32_t C_BETA = 218112;   // beta [64]
constexpr uint32_t C_RB = 218368;     // dbeta partials [4][64] (before them: inverse row norms of the L2-norm prologue)
constexpr uint32_t C_RED = 219392;    // sum_v dX v [64], d(2^G_last) [128]
constexpr uint32_t C_MISC = 220160;   // mbarriers (loads S, P1, P2, raw k/q, products), tmem slot
constexpr uint32_t C_GPB = 220224;    // KDA gate: the dg scan's dbias partials [8 segments][128]
constexpr uint32_t C_GPA = 224320;    //           and dA_log partials [512 threads]
constexpr uint32_t C_SMEM = 226368 + 1024;
static_assert(C_SMEM <= 232448, "one CTA per SM (227 KB)");
constexpr uint32_t LO128 = 16384, LO64 = 8192;  // offsets of the lo twins of 128- and 64-column tiles
struct IntraArgs {
  const __nv_bfloat16 *dO;
  __nv_bfloat16 *dv;  // [B*T][HV][V]
  void *dq, *dk;      // bf16 [B*T][H][K] when HV == H, else fp32 partials [B*T][HV][K]
  float *dg, *dbeta;
  bool partial;
  int *err;
};

// A fragment (16x16, row-major operand) of rows m0.., cols k0.. of a swizzled tile.
__device__ __forceinline__ void lda(uint32_t tile, int R, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31;
  const int row = m0 + (l & 7) + ((l >> 3) & 1) * 8, jj = (k0 >> 3) + (l >> 4);
  ldsm_x4(tile + sw_chunk(row, jj, R), a[0], a[1], a[2], a[3]);
}
// A fragment of the transpose: element (m, k) = tile[k][m]  (rows k0.., cols m0..)
__device__ __forceinline__ void lda_t(uint32_t tile, int R, int m0, int k0, uint32_t (&a)[4]) {
  const int l = threadIdx.x & 31, mi = l >> 3;
  const int row = k0 + (l & 7) + (mi >> 1) * 8, jj = (m0 >> 3) + (mi & 1);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(tile + sw_chunk(row, jj, R)));
}
// B fragments of two n8 tiles: element (k, n) = tile[n][k]  (tile rows n0.., cols k0..)
__device__ __forceinline__ void ldb(uint32_t tile, int R, int n0, int k0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, mi = l >> 3;
  const int row = n0 + (l & 7) + (mi >> 1) * 8, jj = (k0 >> 3) + (mi & 1);
  ldsm_x4(tile + sw_chunk(row, jj, R), b[0], b[1], b[2], b[3]);
}
// B fragments of two n8 tiles: element (k, n) = tile[k][n]  (tile rows k0.., cols n0..)
__device__ __forceinline__ void ldb_t(uint32_t tile, int R, int n0, int k0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31, mi = l >> 3;
  const int row = k0 + (l & 7) + (mi & 1) * 8, jj = (n0 >> 3) + (mi >> 1);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
               : "r"(tile + sw_chunk(row, jj, R)));
}
// Store (a, b) as hi = bf16(x), lo = bf16(x - hi) at element (r, c) of a tile and its lo twin.
__device__ __forceinline__ void st_split2(unsigned char *tile, uint32_t lo_off, int r, int c, int R, float a,
                                          float b) {
  const uint32_t hi = pack_bf16(a, b);
  const float2 h = unpack_bf16(hi);
  const uint32_t off = sw_off(r, c, R);
  *reinterpret_cast<uint32_t *>(tile + off) = hi;
  *reinterpret_cast<uint32_t *>(tile + lo_off + off) = pack_bf16(a - h.x, b - h.y);
}
__device__ __forceinline__ void split8(const float (&x)[8], uint4 &hi, uint4 &lo) {
  hi = pack8(x);
  float h[8], l[8];
  unpack8(hi, h);
#pragma unroll
  for (int e = 0; e < 8; ++e) l[e] = x[e] - h[e];
  lo = pack8(l);
}
// acc += a * b  with a, b each given as (hi, lo): hi*hi + hi*lo + lo*hi
__device__ __forceinline__ void mma3(float (&acc)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma16816(acc, ah, bh0, bh1);
  mma16816(acc, ah, bl0, bl1);
  mma16816(acc, al, bh0, bh1);
}

constexpr int kCT = 512;  // 16 warps: the chain is latency-bound, so more warps hide more of it

// Slot s of the chunk-major (chunk, value head) list; false past the valid
// chunks (the chunk table lists them first).
struct Slot {
  int t0, len, j, h;
  size_t slot;
};
// Which slots a launch walks: all of them, or the list another launch left
// (status word 5: slots whose chunk decay span is too wide for the
// chunk-reference kernel; word 4: slots with a 16-token block too wide for the
// block-reference kernel).  s indexes that list (nlist entries) in list mode.
enum SlotSource { kAllSlots = 0, kChunkWideList = 1, kFixList = 2 };
template <int kSrc>
__device__ __forceinline__ int slot_list_count(const Workspace &W) {
  return kSrc == kAllSlots ? 0 : *(volatile const int *)(W.flags + (kSrc == kFixList ? 4 : 5));
}
// Branch-free in the all-slots mode, so the chunk-table load is only waited
// for where the slot is first used.
template <int kSrc>
__device__ __forceinline__ bool get_slot(const Problem &P, const Workspace &W, int64_t s, int nlist, Slot &o) {
  if (kSrc != kAllSlots) {
    if (s >= nlist) return false;
    s = (kSrc == kFixList ? W.wide_grad : W.wide_cgrad)[s];
  }
  const bool in = s < (int64_t)P.NC * P.HV;
  const int c = in ? (int)(s / P.HV) : 0;
  const int4 ch = W.chunk[c];
  o.j = (int)(s - (int64_t)c * P.HV);
  o.h = o.j / (P.HV / P.H);
  o.t0 = ch.y;
  o.len = ch.z;
  o.slot = (size_t)s;
  return in && ch.x >= 0;
}

// A slot's inputs arrive in three groups of bulk / TMA copies, each into tiles
// that die at a different point of the previous slot's work:
//   P1 (after the pairwise chains): dh', v, A, h columns 64..127 -> the dAqk^T, X, T, A and dL tiles
//   P2 (after the assembly):        dO, dD columns 64..127, h columns 0..63 -> the Kc tile
//   S  (once the dg scan holds its parked dG in registers): X^T, D^T, dX, dO and dD
//                                   columns 0..63, dX columns 64..127 -> the Kr, Qr tiles
// (G and beta follow P2 by cp.async from every thread.)  The stacked
// [dX; dO; dD] operand is two 64-column sub-tiles of 192 rows; h and dh' are
// the saved swizzled tiles, two 64-column halves each.  Inside the slot loop
// thread 0 posts a group's byte count and lane 0 of warps 1.. issue one copy
// each, so no warp stalls for a whole group's issue (an mbarrier's
// transaction count may run below zero until the count is posted).
constexpr uint32_t kBytesS = 2 * 16384u + 4 * 8192u, kBytesP1 = 32768u + 16384u + 8192u + 16384u,
                   kBytesP2 = 2 * 8192u + 16384u;
constexpr int kCopiesS = 6, kCopiesP1 = 4, kCopiesP2 = 3;
// X^T, D^T, h, dh', [dX; dO; dD], v, A: every operand once
static_assert(kBytesS + kBytesP1 + kBytesP2 == 2 * 16384u + 2 * 32768u + 49152u + 16384u + 8192u, "group sizes");
__device__ __forceinline__ void copy_s(int i, uint32_t sbase, const Workspace &W, const TmaMaps &maps, const Slot &q,
                                       uint64_t *bar) {
  const unsigned char *dx = reinterpret_cast<const unsigned char *>(W.tc_dx + q.slot * kC * kD);
  const unsigned char *dd = reinterpret_cast<const unsigned char *>(W.tc_dd + q.slot * kC * kD);
  switch (i) {
    case 0: bulk_load(sbase + I_XT, W.tc_xt + q.slot * 16384, 16384u, bar); break;
    case 1: bulk_load(sbase + I_DT, W.tc_dt + q.slot * 16384, 16384u, bar); break;
    case 2: bulk_load(sbase + I_STK, dx, 8192u, bar); break;                        // dX: rows 0..63, sub-tile 0
    case 3: bulk_load(sbase + I_STK + 192 * 128, dx + 8192, 8192u, bar); break;     //                 sub-tile 1
    case 4: tma_load3(sbase + I_STK + 64 * 128, &maps.d, 0, q.j, q.t0, bar); break;  // dO: rows 64..127, sub-tile 0
    default: bulk_load(sbase + I_STK + 128 * 128, dd, 8192u, bar); break;           // dD: rows 128..191, sub-tile 0
  }
}
__device__ __forceinline__ void copy_p1(int i, uint32_t sbase, const Workspace &W, const TmaMaps &maps,
                                        const Slot &q, uint64_t *bar) {
  switch (i) {
    case 0: bulk_load(sbase + I_DH, W.tc_dh + q.slot * kD * kD, 32768u, bar); break;
    case 1: tma_tile(sbase + I_V, &maps.v, q.j, q.t0, bar); break;
    case 2: bulk_load(sbase + C_A, W.tc_tiles + q.slot * kTileRecord + kRecAM, 8192u, bar); break;
    default:
      bulk_load(sbase + I_H + 16384, reinterpret_cast<const unsigned char *>(W.tc_hs + q.slot * kD * kD) + 16384,
                16384u, bar);
      break;
  }
}
__device__ __forceinline__ void copy_p2(int i, uint32_t sbase, const Workspace &W, const TmaMaps &maps,
                                        const Slot &q, uint64_t *bar) {
  switch (i) {
    case 0: tma_load3(sbase + I_STK + 256 * 128, &maps.d, 64, q.j, q.t0, bar); break;  // dO: rows 64..127, sub-tile 1
    case 1:
      bulk_load(sbase + I_STK + 320 * 128, reinterpret_cast<const unsigned char *>(W.tc_dd + q.slot * kC * kD) + 8192,
                8192u, bar);  // dD, sub-tile 1
      break;
    default: bulk_load(sbase + I_H, W.tc_hs + q.slot * kD * kD, 16384u, bar); break;
  }
}
// G rows (zero past len) and beta of a slot, cp.async from every thread; a
// scalar gate (one decay per token) is repeated over the 128 channels instead
template <bool kScalarGate>
__device__ __forceinline__ void issue_gate_beta(uint32_t sbase, unsigned char *sm, const Problem &P, float *beta,
                                                const Slot &q) {
  const int tid = threadIdx.x;
  if (kScalarGate) {
    float *G = (float *)(sm + C_G);
    constexpr int kIt = kC * 32 / kCT;  // float4 stores per thread; all loads go out first
    float x[kIt];
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int r = (tid + u * kCT) >> 5;
      x[u] = r < q.len ? P.g[(size_t)(q.t0 + r) * P.HV + q.j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int it = tid + u * kCT, r = it >> 5, c4 = (it & 31) * 4;
      *reinterpret_cast<float4 *>(G + r * kGLD + c4) = make_float4(x[u], x[u], x[u], x[u]);
    }
  } else {
    load_gate<kCT>(sbase + C_G, P.g, q.t0, q.len, P.HV, q.j, P.K);
  }
  if (tid < kC) {
    if (tid < q.len) cp4(smem_u32(beta + tid), P.beta + (size_t)(q.t0 + tid) * P.HV + q.j);
    else beta[tid] = 0.f;
  }
  cp_commit();
}


}  // namespace intra

// The chunk-reference kernel over every slot of the chunk table: it lists the
// slots whose chunk decay span is too wide for it in W.wide_cgrad (status word 5)
// for the block-reference kernel.
cudaError_t launch_intra_chunk(const Problem &P, const GateArgs &ga, const Workspace &W, const intra::IntraArgs &a,
                               const TmaMaps &maps, unsigned grid, cudaStream_t s);

}  // namespace kda
