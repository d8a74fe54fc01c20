// Gradient assembly of the bf16 chunked KDA backward (K = V = 128).
//
// One CTA per (chunk, value head).  From the tensor-core products of the
// per-chunk kernel (dQg, dBk, dKhat, dA, dAqk) it finishes
//   dL   = -tril_{-1}(A^T dA A^T)                 gradient through A = (I + L)^-1
//   the chain through L = beta*KK and Aqk to the keys, queries and gate,
// and assembles dq, dk, dg and dbeta.  With 2^(G_r - G_i) split at 16-token
// block starts exactly as in the forward (rows: e1 = 2^(G_r - G_ref) <= 1,
// columns: e2 = 2^(G_ref - G_i), between blocks D_RI <= 1 on the operand):
//   row side    xr = sum_i dL_ri  Kc_i D_RI,  yr = sum_i dAqk_ri Kc_i D_RI
//   column side xi = sum_r X_ri   Kr_r D_RI,  yi = sum_r dAqk_ri Qr_r D_RI   (X = beta dL)
// on 16x16 warp MMAs, then per element (Gamma = 2^G, khat = 2^(G_last - G)):
//   dq~ = dQg Gamma + e1 yr
//   dk  = dKhat khat + beta Gamma dBk + beta e1 xr + e2 (xi + yi)
//   dG  = ln2 [dQg q~ Gamma - dKhat k khat + beta dBk k Gamma + beta k e1 xr + q~ e1 yr - k e2 (xi + yi)]
//   dG_last += ln2 (sum_r dKhat k khat + 2^G_last d(2^G_last))
//   dbeta   = sum_v dX v + sum_c (dBk k Gamma + k e1 xr)
//   dg = reverse cumsum of dG inside the chunk (G is in log2 units).
// All reductions run in a fixed order: the result is bitwise reproducible.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

// shared memory map (bytes from a 1024-aligned base).  "hi/lo" tiles hold a
// value as the sum of two bf16 numbers, so warp MMAs over hi*hi + hi*lo + lo*hi
// keep ~16 mantissa bits: the pairwise terms below sum to zero over a chunk and
// dg accumulates them, so their rounding must stay far below the bf16 level.
constexpr uint32_t C_G = 0;          // G fp32 [64][132]
constexpr uint32_t C_VEC = 33792;    // vectors (20 x 128 fp32)
constexpr uint32_t C_BETA = 44032;   // beta [64]
constexpr uint32_t C_RB = 44288;     // dbeta partials [4][64]
constexpr uint32_t C_RC = 45312;     // prefetched d(2^G_last) [128] and sum_v dX v [64]
constexpr uint32_t C_KR = 47104;     // Kr  hi [64][128] | lo (+16 KB)
constexpr uint32_t C_QR = 79872;     // Qr  hi | lo
constexpr uint32_t C_KC = 112640;    // Kc  hi | lo
constexpr uint32_t C_A = 145408;     // A   [64 r][64 i] bf16
constexpr uint32_t C_DAB = 153600;   // dA^T [64 i][64 m] hi | lo (+8 KB) -> later dL [64 r][64 i] hi | lo
constexpr uint32_t C_DQK = 169984;   // dAqk^T [64 i][64 r] hi | lo
constexpr uint32_t C_XB = 186368;    // X = beta dL [64 r][64 i] hi | lo
constexpr uint32_t C_T = 202752;     // T = A^T dA [64 r][64 m] hi | lo
constexpr uint32_t LO128 = 16384, LO64 = 8192;
// Product staging for the assembly, in four passes of 32 columns (16 per
// column half), double-buffered: each pass holds dQg, dBk, dKhat as
// [64][32] fp32 tiles with 16-byte chunks XOR-swizzled by row % 8 (8 KB each).
// Buffer 0 lives in the A and T tiles (dead after dL, so pass 0 loads during
// the pairwise chains); buffer 1 in the dL / dAqk tiles (dead after the
// chains).  The dG tiles of a pass and the segment totals of its column scans
// use the rest of the dead chain tiles; d(2^G_last) and sum_v dX v are
// prefetched into the C_RC scratch right after dL.
constexpr uint32_t ST_BYTES = 64 * 32 * 4;        // one staged [64][32] product
constexpr uint32_t C_ST0_QB = C_T;                // pass buffer 0: dQg | dBk (16 KB)
constexpr uint32_t C_ST0_K = C_A;                 //                dKhat (8 KB)
constexpr uint32_t C_ST1 = C_DAB;                 // pass buffer 1: dQg | dBk | dKhat (24 KB)
constexpr uint32_t SQ_LD = 36;                    // row stride (floats) of the dG pass tiles
constexpr uint32_t C_SQ = C_ST1 + 3 * ST_BYTES;   // Q part of dG, one pass [64][SQ_LD]
constexpr uint32_t C_SP = C_SQ + 64 * SQ_LD * 4;  // P part
constexpr uint32_t C_TOT = C_SP + 64 * SQ_LD * 4; // segment totals of Q, P [16][32]; Khat column term [2][4][32]
constexpr uint32_t C_DGL = C_RC;                  // d(2^G_last) [128]
constexpr uint32_t C_DBX = C_RC + 512;            // sum_v dX v [64]
static_assert(C_TOT + (16 + 16 + 8) * 32 * 4 <= C_T, "pass scratch overlaps staging buffer 0");
static_assert(C_RC + 768 <= C_KR, "prefetch scratch overlaps the Kr tile");
// byte offset of element (r, c) of a staged [64][32] product
__device__ __forceinline__ uint32_t st_off(int r, int c) {
  return (uint32_t)r * 128u + ((uint32_t)((c >> 2) ^ (r & 7)) << 4) + (uint32_t)(c & 3) * 4u;
}
constexpr uint32_t C_SMEM = 219136 + 1024;
constexpr float kLn2 = 0.69314718055994530942f;

struct ChainArgs {
  void *dq, *dk;  // bf16 [B*T][H][K] when HV == H, else fp32 partials [B*T][HV][K]
  float *dg, *dbeta;
  bool partial;
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

constexpr int kCT = 512;  // 16 warps: the assembly is latency-bound, so more warps hide more of it

__global__ void __launch_bounds__(kCT, 1) kda_bwd_chain_tc_kernel(Problem P, Workspace W, ChainArgs args) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int c_idx = blockIdx.x, j = blockIdx.y;
  const int4 ch = W.chunk[c_idx];
  if (ch.x < 0) return;
  const int t0 = ch.y, len = ch.z;
  const int HV = P.HV, H = P.H, h = j / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t slot = (size_t)c_idx * HV + j;
  float *G = (float *)(sm + C_G);
  float *vec = (float *)(sm + C_VEC);
  float *beta = (float *)(sm + C_BETA);
  float *rb = (float *)(sm + C_RB);
  const __nv_bfloat16 *kin = (const __nv_bfloat16 *)P.k, *qin = (const __nv_bfloat16 *)P.q;
  constexpr float qscale = 0.08838834764831845f;
  KDA_PT_DECL;

  // ---- loads ----
  load_gate<kCT>(sbase + C_G, P.g, t0, len, HV, j);
  {  // A, saved by the forward recompute in this kernel's swizzled layout
    const unsigned char *src = W.tc_tiles + slot * kTileRecord + kTileRecA;
    for (int it = tid; it < 512; it += kCT) cp16(sbase + C_A + it * 16, src + it * 16);
  }
  if (tid < kC) {
    if (tid < len) cp4(smem_u32(beta + tid), P.beta + (size_t)(t0 + tid) * HV + j);
    else beta[tid] = 0.f;
  }
  // Staged asynchronously in tiles that are written only later, so that no
  // thread waits on a plain global load: dA^T, dAqk^T (fp32) in the Kr tile;
  // raw k, q rows in the lo halves of Kc and Qr -- the decay-tile pass reads
  // each 16-byte chunk there before the same thread overwrites it.
  for (int it = tid; it < kC * 16; it += kCT) {
    cp16(sbase + C_KR + it * 16, W.tc_dat + slot * kC * kC + it * 4);
    cp16(sbase + C_KR + LO128 + it * 16, W.tc_dqkt + slot * kC * kC + it * 4);
  }
  load_rows<kCT>(sbase + C_KC + LO128, kin, t0, len, H, h);
  load_rows<kCT>(sbase + C_QR + LO128, qin, t0, len, H, h);
  cp_commit();
  cp_wait_all();
  __syncthreads();
  for (int it = tid; it < kC * 8; it += kCT) {  // dA^T, dAqk^T fp32 -> hi/lo bf16 tiles
    const int r = it >> 3, jj = it & 7;
    const float *a = (const float *)(sm + C_KR) + r * kC + jj * 8;
    const float *b = (const float *)(sm + C_KR + LO128) + r * kC + jj * 8;
    float x[8], y[8];
#pragma unroll
    for (int e = 0; e < 8; e += 4) {
      *reinterpret_cast<float4 *>(x + e) = *reinterpret_cast<const float4 *>(a + e);
      *reinterpret_cast<float4 *>(y + e) = *reinterpret_cast<const float4 *>(b + e);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)  // dAqk^T[i][r] is a gradient of Aqk only where i <= r
      if (r > jj * 8 + e) y[e] = 0.f;
    const uint32_t off = sw_chunk(r, jj, kC);
    uint4 hi, lo;
    split8(x, hi, lo);
    *reinterpret_cast<uint4 *>(sm + C_DAB + off) = hi;
    *reinterpret_cast<uint4 *>(sm + C_DAB + LO64 + off) = lo;
    split8(y, hi, lo);
    *reinterpret_cast<uint4 *>(sm + C_DQK + off) = hi;
    *reinterpret_cast<uint4 *>(sm + C_DQK + LO64 + off) = lo;
  }
  KDA_PT(0);  // (the barrier after the cumsum also orders the Kr staging reads before the Kr writes)

  // ---- G, block references, decay tiles Kr, Qr, Kc (hi/lo) ----
  if (tid < kD) {
    const int c = tid;
    float s = 0.f;
    float col[kC];
#pragma unroll
    for (int r = 0; r < kC; ++r) col[r] = G[r * kGLD + c];
#pragma unroll
    for (int r = 0; r < kC; ++r) {
      if (r < len) s += col[r];
      col[r] = s;
    }
#pragma unroll
    for (int r = 0; r < kC; ++r) G[r * kGLD + c] = col[r];
    const float gl = s;
    vec[V_GL * kD + c] = gl;
    vec[V_GAML * kD + c] = exp2f(gl);
    float gref[4];
#pragma unroll
    for (int R = 0; R < 4; ++R) {
      gref[R] = (16 * R < len) ? col[16 * R] : gl;
      vec[(V_GREF + R) * kD + c] = gref[R];
      vec[(V_EREF + R) * kD + c] = exp2f(gref[R]);
      vec[(V_LAM + R) * kD + c] = exp2f(gl - gref[R]);
    }
    int p = 0;
#pragma unroll
    for (int R = 1; R < 4; ++R)
#pragma unroll
      for (int I = 0; I < R; ++I) vec[(V_D + p++) * kD + c] = exp2f(gref[R] - gref[I]);
  }
  __syncthreads();
  KDA_PT(1);
  {
    const int jj = tid & 15, c0 = jj * 8, rg = tid >> 4, R = rg >> 3;  // two rows per thread
    float gref[8];
#pragma unroll
    for (int e = 0; e < 8; e += 4)
      *reinterpret_cast<float4 *>(gref + e) = *reinterpret_cast<const float4 *>(vec + (V_GREF + R) * kD + c0 + e);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = rg * 2 + rr;
      const uint32_t off = sw_chunk(r, jj, kC);
      float kv[8], qv[8], o[8], e1[8], e2[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + C_KC + LO128 + off), kv);  // raw k, q (zero past len)
      unpack8(*reinterpret_cast<const uint4 *>(sm + C_QR + LO128 + off), qv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float g = G[r * kGLD + c0 + e];
        e1[e] = exp2f(g - gref[e]);
        e2[e] = exp2f(gref[e] - g);
      }
      uint4 hi, lo;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e1[e];
      split8(o, hi, lo);
      *reinterpret_cast<uint4 *>(sm + C_KR + off) = hi;
      *reinterpret_cast<uint4 *>(sm + C_KR + LO128 + off) = lo;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = qv[e] * qscale * e1[e];
      split8(o, hi, lo);
      *reinterpret_cast<uint4 *>(sm + C_QR + off) = hi;
      *reinterpret_cast<uint4 *>(sm + C_QR + LO128 + off) = lo;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e];
      split8(o, hi, lo);
      *reinterpret_cast<uint4 *>(sm + C_KC + off) = hi;
      *reinterpret_cast<uint4 *>(sm + C_KC + LO128 + off) = lo;
    }
  }
  __syncthreads();

  KDA_PT(2);
  // ---- T = A^T dA  (T[r][m] = sum_i' A[i'][r] dA[i'][m]; dA[i'][m] = dA^T[m][i']) ----
  const int mt = warp >> 2, nq = warp & 3;  // 16-row block, 16-column quarter
  {
    float acc[2][4] = {};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4], bh[4], bl[4];
      lda_t(sbase + C_A, kC, 16 * mt, 16 * s, a);  // element (r, i') = A[i'][r]
      ldb(sbase + C_DAB, kC, 16 * nq, 16 * s, bh);  // element (i', m) = dA^T[m][i']
      ldb(sbase + C_DAB + LO64, kC, 16 * nq, 16 * s, bl);
      mma16816(acc[0], a, bh[0], bh[1]);
      mma16816(acc[0], a, bl[0], bl[1]);
      mma16816(acc[1], a, bh[2], bh[3]);
      mma16816(acc[1], a, bl[2], bl[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * mt + (lane >> 2) + 8 * hh, m = 16 * nq + 8 * nt + (lane & 3) * 2;
        st_split2(sm + C_T, LO64, r, m, kC, acc[nt][2 * hh], acc[nt][2 * hh + 1]);
      }
  }
  __syncthreads();
  KDA_PT(3);
  // ---- dL = -tril_{-1}(T A^T); X = beta dL ----
  {
    float acc[2][4] = {};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t ah[4], al[4], b[4];
      lda(sbase + C_T, kC, 16 * mt, 16 * s, ah);  // element (r, m) = T[r][m]
      lda(sbase + C_T + LO64, kC, 16 * mt, 16 * s, al);
      ldb(sbase + C_A, kC, 16 * nq, 16 * s, b);  // element (m, i) = A[i][m]
      mma16816(acc[0], ah, b[0], b[1]);
      mma16816(acc[0], al, b[0], b[1]);
      mma16816(acc[1], ah, b[2], b[3]);
      mma16816(acc[1], al, b[2], b[3]);
    }
    __syncthreads();  // every warp has read dA^T: its tiles become dL
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * mt + (lane >> 2) + 8 * hh, i = 16 * nq + 8 * nt + (lane & 3) * 2;
        const float d0 = (i < r) ? -acc[nt][2 * hh] : 0.f, d1 = (i + 1 < r) ? -acc[nt][2 * hh + 1] : 0.f;
        st_split2(sm + C_DAB, LO64, r, i, kC, d0, d1);
        st_split2(sm + C_XB, LO64, r, i, kC, beta[r] * d0, beta[r] * d1);
      }
  }
  __syncthreads();
  // Asynchronous loads of product pass g (columns 32 q + 8 g .. +7 of each quarter q) into buffer g & 1.
  auto stage = [&](int g) {
    for (int it = tid; it < 3 * 512; it += kCT) {
      const int prod = it >> 9, w = it & 511, r = w >> 3, q = w & 7;  // q: 16-byte chunk of the 32 columns
      const int gc = 32 * (q >> 1) + 8 * g + 4 * (q & 1);             // first global column of the chunk
      const float *src = (prod == 0 ? W.tc_dqg : prod == 1 ? W.tc_dbk : W.tc_dkh) + (slot * kC + r) * kD + gc;
      const uint32_t base = (g & 1) ? C_ST1 + (uint32_t)prod * ST_BYTES
                                    : (prod < 2 ? C_ST0_QB + (uint32_t)prod * ST_BYTES : C_ST0_K);
      cp16(sbase + base + st_off(r, 4 * q), src);
    }
    cp_commit();
  };
  if (tid < 32) cp16(sbase + C_DGL + tid * 16, W.tc_dgl + slot * kD + tid * 4);
  else if (tid < 48) cp16(sbase + C_DBX + (tid - 32) * 16, W.tc_dbx + slot * kC + (tid - 32) * 4);
  stage(0);  // A and T are dead: pass 0 loads during the pairwise chains

  KDA_PT(4);
  // ---- pairwise chains: warp owns rows 16B..16B+15 (as r and as i), columns ch0 .. ch0+31 ----
  // Block-pair products are formed in a temporary, scaled by the per-channel
  // factor D_RI in fp32, and added to the accumulators.
  const int Bk = warp >> 2, ch0 = 32 * (warp & 3);
  float xr[4][4] = {}, yr[4][4] = {}, xyi[4][4] = {};  // xyi = xi + yi (only their sum is used)
  for (int I = 0; I <= Bk; ++I) {  // row side: R = Bk, I = 0..Bk
    const float *Dv = (I < Bk) ? vec + (V_D + Bk * (Bk - 1) / 2 + I) * kD : nullptr;
    uint32_t aLh[4], aLl[4], aQh[4], aQl[4];
    lda(sbase + C_DAB, kC, 16 * Bk, 16 * I, aLh);  // dL[r][i]
    lda(sbase + C_DAB + LO64, kC, 16 * Bk, 16 * I, aLl);
    lda_t(sbase + C_DQK, kC, 16 * Bk, 16 * I, aQh);  // dAqk[r][i] = dAqk^T[i][r]
    lda_t(sbase + C_DQK + LO64, kC, 16 * Bk, 16 * I, aQl);
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      uint32_t bh[4], bl[4];
      ldb_t(sbase + C_KC, kC, ch0 + 16 * nb, 16 * I, bh);  // element (i, c) = Kc[i][c]
      ldb_t(sbase + C_KC + LO128, kC, ch0 + 16 * nb, 16 * I, bl);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float tx[4] = {}, ty[4] = {};
        mma3(tx, aLh, aLl, bh[2 * t], bh[2 * t + 1], bl[2 * t], bl[2 * t + 1]);
        mma3(ty, aQh, aQl, bh[2 * t], bh[2 * t + 1], bl[2 * t], bl[2 * t + 1]);
        const int c = ch0 + 16 * nb + 8 * t + (lane & 3) * 2;
        const float d0 = Dv ? Dv[c] : 1.f, d1 = Dv ? Dv[c + 1] : 1.f;
        float(&X)[4] = xr[2 * nb + t];
        float(&Y)[4] = yr[2 * nb + t];
        X[0] = fmaf(d0, tx[0], X[0]); X[1] = fmaf(d1, tx[1], X[1]); X[2] = fmaf(d0, tx[2], X[2]); X[3] = fmaf(d1, tx[3], X[3]);
        Y[0] = fmaf(d0, ty[0], Y[0]); Y[1] = fmaf(d1, ty[1], Y[1]); Y[2] = fmaf(d0, ty[2], Y[2]); Y[3] = fmaf(d1, ty[3], Y[3]);
      }
    }
  }
  for (int R = Bk; R < 4; ++R) {  // column side: I = Bk, R = Bk..3
    const float *Dv = (R > Bk) ? vec + (V_D + R * (R - 1) / 2 + Bk) * kD : nullptr;
    uint32_t aXh[4], aXl[4], aQh[4], aQl[4];
    lda_t(sbase + C_XB, kC, 16 * Bk, 16 * R, aXh);  // element (i, r) = X[r][i]
    lda_t(sbase + C_XB + LO64, kC, 16 * Bk, 16 * R, aXl);
    lda(sbase + C_DQK, kC, 16 * Bk, 16 * R, aQh);  // element (i, r) = dAqk^T[i][r]
    lda(sbase + C_DQK + LO64, kC, 16 * Bk, 16 * R, aQl);
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      uint32_t kh[4], kl[4], qh[4], ql[4];
      ldb_t(sbase + C_KR, kC, ch0 + 16 * nb, 16 * R, kh);  // element (r, c) = Kr[r][c]
      ldb_t(sbase + C_KR + LO128, kC, ch0 + 16 * nb, 16 * R, kl);
      ldb_t(sbase + C_QR, kC, ch0 + 16 * nb, 16 * R, qh);
      ldb_t(sbase + C_QR + LO128, kC, ch0 + 16 * nb, 16 * R, ql);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float tx[4] = {};  // X Kr + dAqk Qr of this block pair, before the channel decay
        mma3(tx, aXh, aXl, kh[2 * t], kh[2 * t + 1], kl[2 * t], kl[2 * t + 1]);
        mma3(tx, aQh, aQl, qh[2 * t], qh[2 * t + 1], ql[2 * t], ql[2 * t + 1]);
        const int c = ch0 + 16 * nb + 8 * t + (lane & 3) * 2;
        const float d0 = Dv ? Dv[c] : 1.f, d1 = Dv ? Dv[c + 1] : 1.f;
        float(&X)[4] = xyi[2 * nb + t];
        X[0] = fmaf(d0, tx[0], X[0]); X[1] = fmaf(d1, tx[1], X[1]); X[2] = fmaf(d0, tx[2], X[2]); X[3] = fmaf(d1, tx[3], X[3]);
      }
    }
  }
  __syncthreads();  // every warp is done with the chain tiles: A .. X become the product staging
  KDA_PT(5);

  // ---- assembly (fragment element (r, c)), in four passes of 8 columns per warp ----
  // Raw k and q are not re-read: every term that needs them is a product with
  // a decay factor that the hi/lo tiles Kr = k e1, Qr = q~ e1, Kc = k e2 hold.
  // dg = reverse cumsum of dG over the chunk runs per pass as column scans
  // over 4-row segments with segment totals exchanged in shared memory.
  float *sQ = (float *)(sm + C_SQ), *sP = (float *)(sm + C_SP);
  float *totQ = (float *)(sm + C_TOT), *totP = totQ + 16 * 32;
  const float *dglv = (const float *)(sm + C_DGL), *dbxv = (const float *)(sm + C_DBX);
  const int i8 = lane >> 2, l4 = lane & 3, mid = len >> 1;
  float bpart[2] = {0.f, 0.f};
  stage(1);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (g < 3) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    else cp_wait_all();
    __syncthreads();
    KDA_PT(9);
    float *totC = totP + 16 * 32 + (g & 1) * 4 * 32;  // double-buffered: read after the next pass starts
    const uint32_t bq = (g & 1) ? C_ST1 : C_ST0_QB, bb = bq + ST_BYTES, bk = (g & 1) ? C_ST1 + 2 * ST_BYTES : C_ST0_K;
    {
      float qv[1][2][2], pv[1][2][2], cq[1][2];  // [nt of the pass][hh][u], column sums [nt][u]
#pragma unroll
      for (int ntl = 0; ntl < 1; ++ntl) {
        const int nt = g;
        const int c = ch0 + 8 * nt + 2 * l4;
        const int lc = 8 * (warp & 3) + 2 * l4;  // column in the staging
        const float2 gref2 = *reinterpret_cast<const float2 *>(vec + (V_GREF + Bk) * kD + c);
        const float2 eref2 = *reinterpret_cast<const float2 *>(vec + (V_EREF + Bk) * kD + c);
        const float2 lam2 = *reinterpret_cast<const float2 *>(vec + (V_LAM + Bk) * kD + c);
        cq[ntl][0] = cq[ntl][1] = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * Bk + i8 + 8 * hh;
          const float br = beta[r];
          const uint32_t so = st_off(r, lc);
          const float2 vq = *reinterpret_cast<const float2 *>(sm + bq + so);
          const float2 vb = *reinterpret_cast<const float2 *>(sm + bb + so);
          const float2 vk = *reinterpret_cast<const float2 *>(sm + bk + so);
          const uint32_t to = sw_off(r, c, kC);
          const float2 krh = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KR + to));
          const float2 krl = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KR + LO128 + to));
          const float2 qrh = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_QR + to));
          const float2 qrl = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_QR + LO128 + to));
          const float2 kch = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KC + to));
          const float2 kcl = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KC + LO128 + to));
          const float2 g2 = *reinterpret_cast<const float2 *>(G + r * kGLD + c);
          float dq2[2], dk2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float Kr = u ? krh.y + krl.y : krh.x + krl.x;  // k e1
            const float Qr = u ? qrh.y + qrl.y : qrh.x + qrl.x;  // q~ e1
            const float Kc = u ? kch.y + kcl.y : kch.x + kcl.x;  // k e2
            const float dQg = u ? vq.y : vq.x, dBk = u ? vb.y : vb.x, dKh = u ? vk.y : vk.x;
            const float gg_ = u ? g2.y : g2.x, gref = u ? gref2.y : gref2.x;
            const float eref = u ? eref2.y : eref2.x, lam = u ? lam2.y : lam2.x;
            const float e1 = exp2f(gg_ - gref), e2 = exp2f(gref - gg_);
            const float gam = e1 * eref, kh = e2 * lam;
            const float xR = xr[nt][2 * hh + u], yR = yr[nt][2 * hh + u];
            const float xyI = xyi[nt][2 * hh + u];
            dq2[u] = dQg * gam + e1 * yR;
            dk2[u] = dKh * kh + br * gam * dBk + br * e1 * xR + e2 * xyI;
            // dG = Q + P: P (pairwise decay terms and the Khat term) sums to zero over the chunk
            const bool in = r < len;
            qv[ntl][hh][u] = in ? kLn2 * (dQg * Qr * eref + br * dBk * Kr * eref) : 0.f;
            pv[ntl][hh][u] = in ? kLn2 * (br * Kr * xR + Qr * yR - Kc * xyI - dKh * Kc * lam) : 0.f;
            bpart[hh] += dBk * Kr * eref + Kr * xR;
            cq[ntl][u] += dKh * Kc * lam;
          }
          if (r < len) {
            const size_t tok = (size_t)(t0 + r);
            if (args.partial) {
              float *pq = (float *)args.dq + (tok * HV + j) * kD + c, *pk = (float *)args.dk + (tok * HV + j) * kD + c;
              *reinterpret_cast<float2 *>(pq) = make_float2(dq2[0], dq2[1]);  // scaled in the group reduction
              *reinterpret_cast<float2 *>(pk) = make_float2(dk2[0], dk2[1]);
            } else {
              __nv_bfloat16 *pq = (__nv_bfloat16 *)args.dq + (tok * H + h) * kD + c;
              __nv_bfloat16 *pk = (__nv_bfloat16 *)args.dk + (tok * H + h) * kD + c;
              *reinterpret_cast<uint32_t *>(pq) = pack_bf16(dq2[0] * qscale, dq2[1] * qscale);
              *reinterpret_cast<uint32_t *>(pk) = pack_bf16(dk2[0], dk2[1]);
            }
          }
        }
      }
      KDA_PT(10);
      // dG of this pass's 32 columns -> shared memory, then the column scans
#pragma unroll
      for (int ntl = 0; ntl < 1; ++ntl) {
        const int lc = 8 * (warp & 3) + 2 * l4;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * Bk + i8 + 8 * hh;
          *reinterpret_cast<float2 *>(sQ + r * SQ_LD + lc) = make_float2(qv[ntl][hh][0], qv[ntl][hh][1]);
          *reinterpret_cast<float2 *>(sP + r * SQ_LD + lc) = make_float2(pv[ntl][hh][0], pv[ntl][hh][1]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {  // column sums of dKhat k khat over the warp's 16 rows
          float cs = cq[ntl][u];
          cs += __shfl_xor_sync(0xffffffffu, cs, 4);
          cs += __shfl_xor_sync(0xffffffffu, cs, 8);
          cs += __shfl_xor_sync(0xffffffffu, cs, 16);
          if (i8 == 0) totC[Bk * 32 + lc + u] = cs;
        }
      }
      __syncthreads();  // buffer g & 1 consumed; dG tiles complete
      if (g + 2 < 4) stage(g + 2);
      KDA_PT(11);
      {  // thread: one column of the pass, one 4-row segment (warp = segment)
        const int col = tid & 31, seg = warp;
        const int cc = 32 * (col >> 3) + 8 * g + (col & 7);
        float q8[4], p8[4], tq = 0.f, tp = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          q8[k] = sQ[(4 * seg + k) * SQ_LD + col];
          p8[k] = sP[(4 * seg + k) * SQ_LD + col];
          tq += q8[k];
          tp += p8[k];
        }
        totQ[seg * 32 + col] = tq;
        totP[seg * 32 + col] = tp;
        __syncthreads();
        float aq = 0.f, aps = 0.f, app = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < 16; ++s2) {
          const float a = totQ[s2 * 32 + col], b = totP[s2 * 32 + col];
          if (s2 > seg) { aq += a; aps += b; }
          if (s2 < seg) app += b;
        }
        const float ks = totC[col] + totC[32 + col] + totC[64 + col] + totC[96 + col];
        // dg_t = sum_{s>=t} dG_s: the Q part and the carried-state decay term
        // from the chunk end; the zero-sum P part from whichever end is nearer
        // (sum_{s>=t} P_s = -sum_{s<t} P_s, the Khat column sum counted at the
        // last row), halving the cancelling terms it sums.
        const float carried = kLn2 * vec[V_GAML * kD + cc] * dglv[cc];
        float pre[4];
        pre[0] = app;
#pragma unroll
        for (int k = 1; k < 4; ++k) pre[k] = pre[k - 1] + p8[k - 1];
        float qs = aq, ps = aps + kLn2 * ks;
#pragma unroll
        for (int k = 3; k >= 0; --k) {
          const int r = 4 * seg + k;
          qs += q8[k];
          ps += p8[k];
          if (r < len)
            args.dg[((size_t)(t0 + r) * HV + j) * kD + cc] = qs + carried + (r >= mid ? ps : -pre[k]);
        }
      }
      KDA_PT(12);
    }
  }
  KDA_PT(6);
  // dbeta partials: reduce over the 4 lanes sharing a row, then per column half
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float v = bpart[hh];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    if (l4 == 0) rb[(warp & 3) * kC + 16 * Bk + i8 + 8 * hh] = v;
  }
  __syncthreads();
  KDA_PT(7);
  if (tid < kC && tid < len)
    args.dbeta[(size_t)(t0 + tid) * HV + j] = dbxv[tid] + rb[tid] + rb[kC + tid] + rb[2 * kC + tid] + rb[3 * kC + tid];
  KDA_PT(8);
  KDA_PT_FLUSH;
}

}  // namespace

KDA_PT_EXPORT(kda_debug_chain_phase_cycles)

cudaError_t tc_backward_chain(const Problem &P, const Workspace &W, void *dq, void *dk, float *dg,
                              float *dbeta, cudaStream_t s) {
  if (P.NC == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C_SMEM);
  if (e != cudaSuccess) return e;
  const bool partial = P.HV != P.H;
  ChainArgs a{partial ? (void *)W.dqp : dq, partial ? (void *)W.dkp : dk, dg, dbeta, partial};
  KDA_LAUNCH("kda_bwd_chain_tc", s, kda_bwd_chain_tc_kernel<<<dim3(P.NC, P.HV), kCT, C_SMEM, s>>>(P, W, a));
  return cudaGetLastError();
}

}  // namespace kda
