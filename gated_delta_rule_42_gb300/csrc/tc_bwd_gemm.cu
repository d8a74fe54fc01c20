// Per-chunk tensor-core products of the bf16 chunked KDA backward (K = V = 128).
//
// Persistent: one CTA per SM walks the (chunk, value head) slots with a stride
// of the grid, and the loads of its next slot run while it stores the current
// slot's products.  Inputs per slot: the chunk-start state h and the tiles X^T
// (X = beta v - Bk h) and D^T (the deltas D = A X) from the forward recompute,
// the gradient of the chunk-end state dh', and dD, dX from the reverse scan.
// On tcgen05:
//   [dX; dO] h^T    -> rows 0..63: -dBk, rows 64..127: dQg   (one M=128 product)
//   dKhat^T = dh' D^T                                          (Khat = k 2^(G_last - G))
//   [X; D] [dO; dD]^T -> block (X, dD) = dA^T, block (D, dO) = dAqk^T
// and on the SIMT cores dv = beta dX, the beta gradient through v,
// sum_v dX v, and d(2^G_last) = rowsum(dh' .* h).  The products are stored
// (fp32) for the chain kernel, which finishes dq, dk, dg and dbeta.
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
constexpr uint32_t G_XT = 0;         // X^T [128 v][64 r]  (saved by the forward recompute)
constexpr uint32_t G_DT = 16384;     // D^T [128 v][64 r]  (adjacent: [X; D]^T is one MN-major operand)
constexpr uint32_t G_STK = 32768;    // [dX; dO; dD] [192][128]
constexpr uint32_t G_H = 81920;      // h  [128 c][128 v]
constexpr uint32_t G_DH = 114688;    // dh' [128 c][128 v]
constexpr uint32_t G_V = 147456;     // v  [64 r][128 v]
constexpr uint32_t G_BETA = 163840;  // beta [64]
constexpr uint32_t G_RED = 164096;   // reductions: dbeta_x [64], dGl [128]
constexpr uint32_t G_MISC = 164864;  // mbarrier, tmem slot
constexpr uint32_t G_SMEM = 164928 + 1024;
constexpr uint32_t TMEM_COLS = 512;  // [128,256) S, [256,320) dKhat^T, [384,512) Z

struct GemmArgs {
  const __nv_bfloat16 *dO;
  __nv_bfloat16 *dv;  // output [B*T][HV][V]
  int *err;
};

__global__ void __launch_bounds__(kThr, 1) kda_bwd_gemm_tc_kernel(Problem P, Workspace W, GemmArgs args) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int HV = P.HV;
  const int nslots = P.NC * HV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int lrow = quarter * 32 + lane;  // TMEM lane of this thread
  float *beta = (float *)(sm + G_BETA);
  float *red = (float *)(sm + G_RED);
  uint64_t *bar = (uint64_t *)(sm + G_MISC);
  uint32_t *tslot = (uint32_t *)(sm + G_MISC + 8);
  const __nv_bfloat16 *vin = (const __nv_bfloat16 *)P.v;

  if (tid == 0) {
    bar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
  uint32_t phase = 0;

  // All loads of slot s (chunk entry ch) as one cp.async group.
  auto issue = [&](int s, int4 ch) {
    const int j = s % HV, t0 = ch.y, len = ch.z;
    const size_t slot = (size_t)s;
    const unsigned char *xt = W.tc_xt + slot * 16384, *dt = W.tc_dt + slot * 16384;
    for (int it = tid; it < 1024; it += kThr) {  // X^T, D^T: verbatim (same swizzled layout)
      cp16(sbase + G_XT + it * 16, xt + it * 16);
      cp16(sbase + G_DT + it * 16, dt + it * 16);
    }
    for (int it = tid; it < 128 * 16; it += kThr) {  // h and dh' [128][128], saved swizzled: verbatim
      cp16(sbase + G_H + it * 16, reinterpret_cast<const unsigned char *>(W.tc_hs + slot * kD * kD) + it * 16);
      cp16(sbase + G_DH + it * 16, reinterpret_cast<const unsigned char *>(W.tc_dh + slot * kD * kD) + it * 16);
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
    load_rows(sbase + G_V, vin, t0, len, HV, j);
    if (tid < kC) {
      if (tid < len) cp4(smem_u32(beta + tid), P.beta + (size_t)(t0 + tid) * HV + j);
      else beta[tid] = 0.f;
    }
    cp_commit();
  };

  // Slots are chunk-major; the chunk table ends with unused entries (x < 0),
  // so a CTA stops at its first unused slot.
  int s = blockIdx.x;
  int4 ch = s < nslots ? W.chunk[s / HV] : make_int4(-1, 0, 0, 0);
  if (ch.x >= 0) issue(s, ch);
  while (ch.x >= 0) {
    const int sn = s + gridDim.x;
    const int4 chn = sn < nslots ? W.chunk[sn / HV] : make_int4(-1, 0, 0, 0);
    const int j = s % HV, t0 = ch.y, len = ch.z;
    const size_t slot = (size_t)s;
    cp_wait_all();
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();

    if (tid == 0) {
      // S[i'][c] = sum_v [dX; dO][i'][v] h[c][v]   (M=128, N=128 c, K=128 v)
      const uint32_t id3 = idesc(128, 128, 0, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + 128, desc_k16(sbase + G_STK, k, 192), desc_k16(sbase + G_H, k, kD), id3, k > 0);
      // dKhat^T[c][r] = sum_v dh'[c][v] D[r][v]   (M=128 c, N=64 r, K=128 v)
      const uint32_t id4 = idesc(128, 64, 0, 1), id5 = idesc(128, 128, 1, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + 256, desc_k16(sbase + G_DH, k, kD), desc_mn(sbase + G_DT, k, 8192), id4, k > 0);
      // Z[i'][n'] = sum_v [X; D][i'][v] [dO; dD][n'][v]   (M=128, N=128, K=128 v)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + 384, desc_mn(sbase + G_XT, k, 16384), desc_k16(sbase + G_STK + 64 * 128, k, 192), id5, k > 0);
      commit(bar);
    }
    // meanwhile on the SIMT cores: d(2^G_last)[c] = sum_v dh'[c][v] h[c][v]; dv; sum_v dX v
    if (tid < kD) {
      const int c = tid;
      float acc = 0.f;
#pragma unroll 4
      for (int jj = 0; jj < 16; ++jj) {
        float a[8], b[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + G_H + sw_chunk(c, jj, kD)), a);
        unpack8(*reinterpret_cast<const uint4 *>(sm + G_DH + sw_chunk(c, jj, kD)), b);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(a[e], b[e], acc);
      }
      red[64 + c] = acc;
    }
    for (int r = warp; r < len; r += 8) {  // one warp per row, 4 columns per lane
      const float br = beta[r];
      const int v0 = lane * 4;
      const uint2 xd = *reinterpret_cast<const uint2 *>(sm + G_STK + sw_off(r, v0, 192));
      const uint2 xv = *reinterpret_cast<const uint2 *>(sm + G_V + sw_off(r, v0, kC));
      const float2 d01 = unpack_bf16(xd.x), d23 = unpack_bf16(xd.y);
      const float2 v01 = unpack_bf16(xv.x), v23 = unpack_bf16(xv.y);
      *reinterpret_cast<uint2 *>(args.dv + ((size_t)(t0 + r) * HV + j) * kD + v0) =
          make_uint2(pack_bf16(br * d01.x, br * d01.y), pack_bf16(br * d23.x, br * d23.y));
      float part = d01.x * v01.x + d01.y * v01.y + d23.x * v23.x + d23.y * v23.y;
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) red[r] = part;
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    __syncthreads();  // products in TMEM; every shared tile of this slot is consumed
    if (chn.x >= 0) issue(sn, chn);

    // ---- store the products (overlaps the next slot's loads) ----
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
      // dKhat^T in TMEM (lane c, 64 columns r: warps half 0 -> r 0..31, half 1 -> r 32..63),
      // stored as dKhat [r][c]: one coalesced 128-byte row segment per warp store
      tmem_ld32(tq + 256u + (uint32_t)(32 * half), d);
      float *dk2 = W.tc_dkh + (slot * kC + 32 * half) * kD + lrow;
#pragma unroll
      for (int e = 0; e < 32; ++e) dk2[e * kD] = d[e];
      // Z: lanes 0..63 (i), cols 64..127 (r) = dA^T [i][r]; lanes 64..127, cols 0..63 = dAqk^T [i][r]
      const uint32_t zc = lrow < 64 ? 64u : 0u;
      tmem_ld32(tq + 384u + zc + (uint32_t)(32 * half), d);
      float *za = (lrow < 64 ? W.tc_dat : W.tc_dqkt) + (slot * kC + (lrow & 63)) * kC + 32 * half;
#pragma unroll
      for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4 *>(za + e) = make_float4(d[e], d[e + 1], d[e + 2], d[e + 3]);
    }
    if (tid < kC) W.tc_dbx[slot * kC + tid] = tid < len ? red[tid] : 0.f;
    if (tid < kD) W.tc_dgl[slot * kD + tid] = red[64 + tid];
    fence_before();  // this slot's TMEM reads precede the next slot's products
    s = sn;
    ch = chn;
  }
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
  int sms = 0;
  if ((e = sm_count(&sms)) != cudaSuccess) return e;
  const long long nslots = (long long)P.NC * P.HV;
  const int grid = (int)(nslots < sms ? nslots : sms);
  GemmArgs a{(const __nv_bfloat16 *)dO, (__nv_bfloat16 *)dv, err};
  KDA_LAUNCH("kda_bwd_gemm_tc", s, kda_bwd_gemm_tc_kernel<<<grid, kThr, G_SMEM, s>>>(P, W, a));
  return cudaGetLastError();
}

}  // namespace kda
