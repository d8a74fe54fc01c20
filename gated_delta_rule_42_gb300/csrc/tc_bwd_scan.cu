// Reverse state-gradient scan of the bf16 chunked KDA backward (K = V = 128).
//
// One CTA walks the chunks of one (sequence, value head) from last to first,
// holding dh' -- the gradient of the chunk-END state -- in fp32 registers
// (thread = key channel c, half the value columns), starting from dhT (or 0).
// Per chunk, with the chunk tiles Bk = beta k 2^G, Qg = q~ 2^G, Khat =
// k 2^(G_last - G), Aqk, A and 2^G_last saved by the forward recompute (one
// bulk copy per chunk: the scan reads no q, k, g or beta), on tcgen05:
//   dD^T = dO^T Aqk + dh'^T Khat^T        dD = Aqk^T dO + Khat dh'   (deltas' gradient)
//   dX^T = dD^T A                         dX = A^T dD                (through A = (I+L)^-1)
//   dh  <- diag(2^G_last) dh' + Qg^T dO - Bk^T dX                    (gradient of the chunk-start state)
// The last line is the reverse recurrence of FLA's bwd_dhu ("[Fix] Use unit KDA
// gate scale when A_log is omitted", fla-org/flash-linear-attention PR #1294,
// commit log: "the kernel's reverse state-gradient recurrence").  Every
// operand is read straight from the row-major tiles through K- or MN-major
// descriptors.  For the per-chunk gradient kernel the scan saves, per chunk,
// with bulk stores from shared memory: dh' (bf16 [K][V]) and dD, dX (bf16
// [64][V]), all in the swizzled operand layout; at the start of the sequence
// it writes dh0 (fp32).
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

constexpr uint32_t U_DH = 0, U_DDT = 32768, U_NDX = 49152;  // phase (c) use of the union
constexpr uint32_t TMEM_COLS = 256;  // [0,64) dD^T, [64,128) dX^T, [128,256) dh update

__global__ void __launch_bounds__(kThr, 1)
kda_bwd_scan_tc_kernel(Problem P, Workspace W, const __nv_bfloat16 *__restrict__ dO,
                       const float *__restrict__ dhT, float *__restrict__ dh0, int *err) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  float *vec = (float *)(sm + OFF_VEC);
  uint64_t *bar = (uint64_t *)(sm + OFF_MISC);
  uint32_t *tslot = (uint32_t *)(sm + OFF_MISC + 8);
  uint64_t *bar_t = (uint64_t *)(sm + OFF_MISC + 16);
  unsigned char *U = sm + OFF_U;

  const int n = blockIdx.x, j = blockIdx.y;
  const int HV = P.HV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, vhalf = warp >> 2;
  const int cown = quarter * 32 + lane;
  const int4 si = W.seq[n];

  if (tid == 0) {
    bar_init(bar, 1);
    bar_init(bar_t, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
  uint32_t phase = 0, t_par = 0;

  float dreg[64];  // dh'[cown][64 * vhalf + x]
  {
    const size_t base = (((size_t)n * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4) {
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (dhT != nullptr) t = *reinterpret_cast<const float4 *>(dhT + base + x);
      dreg[x] = t.x; dreg[x + 1] = t.y; dreg[x + 2] = t.z; dreg[x + 3] = t.w;
    }
  }

  // The chunk tiles Bk, Qg, Khat, Aqk, A and 2^G_last saved by the forward
  // recompute: one bulk copy of the 64 KB record (the Bk .. A region of the
  // shared-memory map, same swizzled layout) and one of the 512-byte vector.
  auto load_tiles = [&](int cidx) {
    const unsigned char *src = W.tc_tiles + ((size_t)cidx * HV + j) * kTileRecord;
    mbar_expect_tx(bar_t, 65536u + 512u);
    bulk_load(sbase + OFF_BK, src, 65536u, bar_t);
    bulk_load(smem_u32(vec + V_GAML * kD), src + 65536, 512u, bar_t);
  };
  if (si.w > 0) {
    const int2 chl = chunk_span(si, si.w - 1);
    if (tid == 0) load_tiles(si.z + si.w - 1);
    load_rows(sbase + OFF_VRAW, dO, chl.x, chl.y, HV, j);
    cp_commit();
  }

  for (int ci = si.w - 1; ci >= 0; --ci) {
    const int cidx = si.z + ci;
    const size_t slot = (size_t)cidx * HV + j;
    cp_wait_all();  // dO
    if (tid == 0) bulk_wait_read();  // the previous chunk's saved tiles have left shared memory
    bar_wait(bar_t, t_par, err);
    t_par ^= 1;
    __syncthreads();

    // ---------------- (c) ----------------
    {
      unsigned char *DH = U + U_DH;  // dh' [c][v], swizzled
#pragma unroll
      for (int x8 = 0; x8 < 8; ++x8) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = dreg[8 * x8 + e];
        *reinterpret_cast<uint4 *>(DH + sw_chunk(cown, 8 * vhalf + x8, kD)) = pack8(t);
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t aDH = sbase + OFF_U + U_DH, aDDT = sbase + OFF_U + U_DDT, aNDX = sbase + OFF_U + U_NDX;
    if (tid == 0) {  // dh' for the per-chunk kernel (its swizzled operand layout)
      bulk_store(W.tc_dh + slot * kD * kD, aDH, 32768u);
      bulk_commit();
    }
    if (tid == 0) {
      // dD^T[v][r] = sum_i dO[i][v] Aqk[i][r] + sum_c dh'[c][v] Khat[r][c]   (M=128 v, N=64 r)
      const uint32_t id1 = idesc(128, 64, 1, 1), id2 = idesc(128, 64, 1, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem, desc_mn(sbase + OFF_VRAW, s, 8192), desc_mn(sbase + OFF_AQK, s, 8192), id1, s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma(tmem, desc_mn(aDH, s, 16384), desc_k16(sbase + OFF_KH, s, kC), id2, 1);
      commit(bar);
    }
    bar_wait(bar, phase, err);
    phase ^= 1;
    fence_after();
    {  // dD^T -> bf16 tile [v][r]; dD -> workspace, row-major [r][v]
      const int v = cown, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tq + (uint32_t)r0, d);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = d[q8 * 8 + e];
        *reinterpret_cast<uint4 *>(U + U_DDT + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e)  // [r][v] in the swizzled K-major operand layout
        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_KRAW + sw_off(r0 + e, v, kC)) = __float2bfloat16_rn(d[e]);
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {  // dD [r][v] (swizzled operand layout) for the per-chunk kernel
      bulk_store(W.tc_dd + slot * kC * kD, sbase + OFF_KRAW, 16384u);
      bulk_commit();
    }
    if (tid == 0) {  // dX^T[v][i] = sum_r dD^T[v][r] A[r][i]   (M=128 v, N=64 i, K=64 r)
      const uint32_t id = idesc(128, 64, 0, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma(tmem + 64, desc_k16(aDDT, s, kD), desc_mn(sbase + OFF_AM, s, 8192), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, err);
    phase ^= 1;
    fence_after();
    {  // -dX^T -> bf16 tile [v][i]; dX -> workspace, row-major [i][v]
      const int v = cown, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tq + 64u + (uint32_t)r0, d);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = -d[q8 * 8 + e];
        *reinterpret_cast<uint4 *>(U + U_NDX + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
      }
#pragma unroll
      for (int e = 0; e < 32; ++e)  // [i][v] in the swizzled K-major operand layout
        *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_QRAW + sw_off(r0 + e, v, kC)) = __float2bfloat16_rn(d[e]);
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {  // dX [i][v] (swizzled operand layout) for the per-chunk kernel
      bulk_store(W.tc_dx + slot * kC * kD, sbase + OFF_QRAW, 16384u);
      bulk_commit();
    }
    if (tid == 0) {
      // U[c][v] = sum_r Qg[r][c] dO[r][v] - sum_r Bk[r][c] dX[r][v]   (M=128 c, N=128 v, K=64 r)
      const uint32_t id1 = idesc(128, 128, 1, 1), id2 = idesc(128, 128, 1, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_mn(sbase + OFF_QG, s, 8192), desc_mn(sbase + OFF_VRAW, s, 8192), id1, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_mn(sbase + OFF_BK, s, 8192), desc_k16(aNDX, s, kD), id2, 1);
      commit(bar);
    }
    bar_wait(bar, phase, err);
    phase ^= 1;
    fence_after();
    {
      const float gl = vec[V_GAML * kD + cown];
      float d[32];
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        tmem_ld32(tq + 128u + (uint32_t)(64 * vhalf + 32 * hx), d);
#pragma unroll
        for (int e = 0; e < 32; ++e) dreg[32 * hx + e] = fmaf(gl, dreg[32 * hx + e], d[e]);
      }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (ci > 0) {  // dO, the tiles and 2^G_last of this chunk consumed
      const int2 pv = chunk_span(si, ci - 1);
      if (tid == 0) {
        fence_async_smem();
        load_tiles(cidx - 1);
      }
      load_rows(sbase + OFF_VRAW, dO, pv.x, pv.y, HV, j);
      cp_commit();
    }
  }

  if (dh0 != nullptr) {
    float *dst = dh0 + (((size_t)n * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4)
      *reinterpret_cast<float4 *>(dst + x) = make_float4(dreg[x], dreg[x + 1], dreg[x + 2], dreg[x + 3]);
  }
  if (tid == 0) bulk_wait_all();  // the saved tiles are in global memory before the CTA exits
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_free(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t tc_backward_scan(const Problem &P, const Workspace &W, const void *dO, const float *dhT,
                             float *dh0, int *err, cudaStream_t s) {
  if (P.N == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  KDA_LAUNCH("kda_bwd_scan_tc", s,
             kda_bwd_scan_tc_kernel<<<dim3(P.N, P.HV), kThr, SMEM_BYTES, s>>>(
                 P, W, (const __nv_bfloat16 *)dO, dhT, dh0, err));
  return cudaGetLastError();
}

}  // namespace kda
