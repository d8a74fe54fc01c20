// Per-chunk tensor-core products of the bf16 chunked KDA backward (K = V = 128).
//
// One CTA per (chunk, value head), all chunks in parallel.  Inputs: the
// chunk-start state h (from the forward recompute), the gradient of the
// chunk-end state dh', and dD, dX, A from the reverse scan.  On tcgen05:
//   X^T  = (beta v)^T - h^T Bk^T                     recompute X = beta v - Bk h
//   D^T  = X^T A^T                                   recompute the deltas D = A X
//   [dX; dO] h^T    -> rows 0..63: -dBk, rows 64..127: dQg   (one M=128 product)
//   dKhat^T = dh' D^T                                          (Khat = k 2^(G_last - G))
//   [X; D] [dO; dD]^T -> block (X, dD) = dA^T, block (D, dO) = dAqk^T
// and on the SIMT cores dv = beta dX, the beta gradient through v,
// sum_v dX v, and d(2^G_last) = rowsum(dh' .* h).  The products are stored
// (bf16 / fp32) for the chain kernel, which finishes dq, dk, dg and dbeta.
// These are the intra-chunk backward products of FLA's chunk_bwd_dqkwg /
// chunk_bwd_dv_local / prepare_wy_repr_bwd ("[Fix] Use unit KDA gate scale when
// A_log is omitted", fla-org/flash-linear-attention PR #1294, commit log),
// stacked so that every tensor-core product has M = 128.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t G_K = 0;          // k [64][128] bf16
constexpr uint32_t G_G = 16384;      // g -> G fp32 [64][132]
constexpr uint32_t G_BETA = 50176;   // beta [64]
constexpr uint32_t G_RED = 50432;    // reductions: dbeta_x [64], dGl [128]
constexpr uint32_t G_MISC = 51200;   // mbarrier, tmem slot
constexpr uint32_t G_BK = 52224;     // Bk [64][128]  -> later X^T [128 v][64 r]
constexpr uint32_t G_AM = 68608;     // A [64][64]    -> later D^T [128 v][64 r]
constexpr uint32_t G_STK = 84992;    // [dX; dO; dD] [192][128]
constexpr uint32_t G_H = 134144;     // h  [128 c][128 v]
constexpr uint32_t G_DH = 166912;    // dh' [128 c][128 v]
constexpr uint32_t G_SMEM = 199680 + 1024;
constexpr uint32_t TMEM_COLS = 512;  // [0,64) X'^T, [64,128) D^T, [128,256) S, [256,320) dKhat^T, [384,512) Z

struct GemmArgs {
  const __nv_bfloat16 *dO;
  __nv_bfloat16 *dv;  // output [B*T][HV][V]
  int *err;
};

__global__ void __launch_bounds__(kThr, 1) kda_bwd_gemm_tc_kernel(Problem P, Workspace W, GemmArgs args) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int c_idx = blockIdx.x, j = blockIdx.y;
  const int4 ch = W.chunk[c_idx];
  if (ch.x < 0) return;
  const int t0 = ch.y, len = ch.z;
  const int HV = P.HV, h = j / (HV / P.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int lrow = quarter * 32 + lane;  // TMEM lane of this thread
  const size_t slot = (size_t)c_idx * HV + j;
  float *G = (float *)(sm + G_G);
  float *beta = (float *)(sm + G_BETA);
  float *red = (float *)(sm + G_RED);
  uint64_t *bar = (uint64_t *)(sm + G_MISC);
  uint32_t *tslot = (uint32_t *)(sm + G_MISC + 8);
  const __nv_bfloat16 *vin = (const __nv_bfloat16 *)P.v;

  // ---- loads ----
  load_rows(sbase + G_K, (const __nv_bfloat16 *)P.k, t0, len, P.H, h);
  load_gate(sbase + G_G, P.g, t0, len, HV, j);
  for (int it = tid; it < 128 * 16; it += kThr) {  // h and dh' [128][128]
    const int r = it >> 4, jj = it & 15;
    cp16(sbase + G_H + sw_chunk(r, jj, kD), W.tc_hs + (slot * kD + r) * kD + jj * 8);
    cp16(sbase + G_DH + sw_chunk(r, jj, kD), W.tc_dh + (slot * kD + r) * kD + jj * 8);
  }
  for (int it = tid; it < 192 * 16; it += kThr) {  // [dX; dO; dD]
    const int r = it >> 4, jj = it & 15;
    const uint32_t dst = sbase + G_STK + sw_chunk(r, jj, 192);
    const int rr = r & 63;
    if (r < 64) cp16(dst, W.tc_dx + (slot * kC + rr) * kD + jj * 8);
    else if (r >= 128) cp16(dst, W.tc_dd + (slot * kC + rr) * kD + jj * 8);
    else if (rr < len) cp16(dst, args.dO + ((size_t)(t0 + rr) * HV + j) * kD + jj * 8);
    else st_zero16(dst);
  }
  for (int it = tid; it < kC * 8; it += kThr) {  // A [64][64]
    const int r = it >> 3, jj = it & 7;
    cp16(sbase + G_AM + sw_chunk(r, jj, kC), W.tc_A + (slot * kC + r) * kC + jj * 8);
  }
  cp_commit();
  if (tid < kC) beta[tid] = tid < len ? P.beta[(size_t)(t0 + tid) * HV + j] : 0.f;
  if (tid == 0) {
    bar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  cp_wait_all();
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
  uint32_t phase = 0;

  // ---- G and Bk = beta k 2^G ----
  if (tid < kD) {
    const int c = tid;
    float s = 0.f;
    for (int r = 0; r < kC; ++r) {
      if (r < len) s += G[r * kGLD + c];
      G[r * kGLD + c] = s;
    }
  }
  __syncthreads();
  for (int it = tid; it < kC * 16; it += kThr) {
    const int r = it >> 4, jj = it & 15;
    const uint32_t off = sw_chunk(r, jj, kC);
    float kv[8], o[8];
    unpack8(*reinterpret_cast<const uint4 *>(sm + G_K + off), kv);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = beta[r] * kv[e] * exp2f(G[r * kGLD + jj * 8 + e]);
    *reinterpret_cast<uint4 *>(sm + G_BK + off) = pack8(o);
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();

  // ---- X'^T = h^T Bk^T and S = [dX; dO] h^T ----
  if (tid == 0) {
    const uint32_t id1 = idesc(128, 64, 1, 0), id3 = idesc(128, 128, 0, 0);
#pragma unroll
    for (int s = 0; s < 8; ++s) mma(tmem, desc_mn(sbase + G_H, s, 16384), desc_k16(sbase + G_BK, s, kC), id1, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      mma(tmem + 128, desc_k16(sbase + G_STK, s, 192), desc_k16(sbase + G_H, s, kD), id3, s > 0);
    commit(bar);
  }
  bar_wait(bar, phase, args.err);
  phase ^= 1;
  fence_after();
  {  // X^T[v][r] = beta_r v[r][v] - X'^T[v][r]  -> tile [v][r] in the Bk slot
    const int v = lrow, r0 = 32 * half;
    float d[32];
    tmem_ld32(tq + (uint32_t)r0, d);
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int r = r0 + q8 * 8 + e;
        const float vv = r < len ? __bfloat162float(vin[((size_t)(t0 + r) * HV + j) * kD + v]) : 0.f;
        x[e] = beta[r] * vv - d[q8 * 8 + e];
      }
      *reinterpret_cast<uint4 *>(sm + G_BK + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
    }
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  if (tid == 0) {  // D^T = X^T A^T  (M=128 v, N=64 r, K=64 i)
    const uint32_t id = idesc(128, 64, 0, 0);
#pragma unroll
    for (int s = 0; s < 4; ++s) mma(tmem + 64, desc_k16(sbase + G_BK, s, kD), desc_k16(sbase + G_AM, s, kC), id, s > 0);
    commit(bar);
  }
  bar_wait(bar, phase, args.err);
  phase ^= 1;
  fence_after();
  {  // D^T -> tile [v][r] in the A slot (adjacent to X^T)
    const int v = lrow, r0 = 32 * half;
    float d[32];
    tmem_ld32(tq + 64u + (uint32_t)r0, d);
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = d[q8 * 8 + e];
      *reinterpret_cast<uint4 *>(sm + G_AM + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
    }
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  if (tid == 0) {
    // dKhat^T[c][r] = sum_v dh'[c][v] D[r][v]   (M=128 c, N=64 r, K=128 v)
    const uint32_t id4 = idesc(128, 64, 0, 1), id5 = idesc(128, 128, 1, 0);
#pragma unroll
    for (int s = 0; s < 8; ++s) mma(tmem + 256, desc_k16(sbase + G_DH, s, kD), desc_mn(sbase + G_AM, s, 8192), id4, s > 0);
    // Z[i'][n'] = sum_v [X; D][i'][v] [dO; dD][n'][v]   (M=128, N=128, K=128 v)
#pragma unroll
    for (int s = 0; s < 8; ++s)
      mma(tmem + 384, desc_mn(sbase + G_BK, s, 16384), desc_k16(sbase + G_STK + 64 * 128, s, 192), id5, s > 0);
    commit(bar);
  }
  // meanwhile on the SIMT cores: d(2^G_last)[c] = sum_v dh'[c][v] h[c][v]; dv; sum_v dX v
  if (tid < kD) {
    const int c = tid;
    float s = 0.f;
#pragma unroll 4
    for (int jj = 0; jj < 16; ++jj) {
      float a[8], b[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + G_H + sw_chunk(c, jj, kD)), a);
      unpack8(*reinterpret_cast<const uint4 *>(sm + G_DH + sw_chunk(c, jj, kD)), b);
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fmaf(a[e], b[e], s);
    }
    red[64 + c] = s;
  }
  for (int r = warp; r < len; r += 8) {  // one warp per row: dv = beta dX, sum_v dX v
    const float br = beta[r];
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = lane * 4 + q;
      const float dx = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + G_STK + sw_off(r, v, 192)));
      const size_t e = ((size_t)(t0 + r) * HV + j) * kD + v;
      args.dv[e] = __float2bfloat16_rn(br * dx);
      part = fmaf(dx, __bfloat162float(vin[e]), part);
    }
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[r] = part;
  }
  bar_wait(bar, phase, args.err);
  phase ^= 1;
  fence_after();
  __syncthreads();
  // ---- store the products ----
  {
    // S: lanes 0..63 = dX h^T = -dBk [i][c], lanes 64..127 = dQg [r][c]
    const int r = lrow & 63;
    float *dst = (lrow < 64 ? W.tc_dbk : W.tc_dqg) + (slot * kC + r) * kD + 64 * half;
    const float sg = lrow < 64 ? -1.f : 1.f;
    float d[32];
#pragma unroll
    for (int hx = 0; hx < 2; ++hx) {
      tmem_ld32(tq + 128u + (uint32_t)(64 * half + 32 * hx), d);
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4 *>(dst + 32 * hx + e) =
            make_float4(sg * d[e], sg * d[e + 1], sg * d[e + 2], sg * d[e + 3]);
    }
    // dKhat^T [c][r] (lane c, 64 columns r: warps half 0 -> r 0..31, half 1 -> r 32..63)
    tmem_ld32(tq + 256u + (uint32_t)(32 * half), d);
    float *dk2 = W.tc_dkh + (slot * kD + lrow) * kC + 32 * half;
#pragma unroll
    for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4 *>(dk2 + e) = make_float4(d[e], d[e + 1], d[e + 2], d[e + 3]);
    // Z: lanes 0..63 (i), cols 64..127 (r) = dA^T [i][r]; lanes 64..127, cols 0..63 = dAqk^T [i][r]
    const uint32_t zc = lrow < 64 ? 64u : 0u;
    tmem_ld32(tq + 384u + zc + (uint32_t)(32 * half), d);
    float *za = (lrow < 64 ? W.tc_dat : W.tc_dqkt) + (slot * kC + (lrow & 63)) * kC + 32 * half;
#pragma unroll
    for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4 *>(za + e) = make_float4(d[e], d[e + 1], d[e + 2], d[e + 3]);
  }
  if (tid < kC) W.tc_dbx[slot * kC + tid] = tid < len ? red[tid] : 0.f;
  if (tid < kD) W.tc_dgl[slot * kD + tid] = red[64 + tid];
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_free(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t tc_backward_gemm(const Problem &P, const Workspace &W, const void *dO, void *dv, int *err,
                             cudaStream_t s) {
  if (P.NC == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)G_SMEM);
  if (e != cudaSuccess) return e;
  GemmArgs a{(const __nv_bfloat16 *)dO, (__nv_bfloat16 *)dv, err};
  KDA_LAUNCH("kda_bwd_gemm_tc", s, kda_bwd_gemm_tc_kernel<<<dim3(P.NC, P.HV), kThr, G_SMEM, s>>>(P, W, a));
  return cudaGetLastError();
}

}  // namespace kda
