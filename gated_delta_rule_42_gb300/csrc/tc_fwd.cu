// Fused bf16 chunked KDA forward on the sm_103a tensor cores (K = V = 128).
//
// One CTA walks the chunks of one (sequence, value head) in order, keeping the
// fp32 state h[K][V] in registers (thread = key channel c, half the value
// columns).  Per 64-token chunk, after the V-independent phases (a) and (b) of
// tc_common.cuh, the state chain runs on tcgen05 (operands in shared memory,
// fp32 accumulators in tensor memory):
//   X^T = (beta v)^T - h^T Bk^T          X = beta v - (beta k 2^G) h
//   D^T = X^T A^T                         D = u - w h, the chunk's deltas
//   O^T = h^T Qg^T + D^T Aqk^T            o = (q~ 2^G) h + Aqk D
//   h  <- diag(2^G_last) h + Khat^T D     the carried state
// h and Khat are stored row-major and read as MN-major operands, so no tile is
// ever transposed.  This is the chunk decomposition of the FLA KDA/GDN pipeline
// (kkt + solve_tril + recompute_w_u + fwd_h + fwd_o, named in the commit log of
// "[Fix] Use unit KDA gate scale when A_log is omitted", fla-org/
// flash-linear-attention PR #1294) fused into one pass, with the [K, V] fp32
// state held on chip across chunks as in the recurrent_kda kernel of "kda in
// torchtitan (training)" (pytorch/torchtitan PR #4164).
//
// In "states" mode (no output) the kernel saves, per chunk, what the backward
// needs from the forward recompute, as bulk copies of its shared-memory tiles
// (swizzled, verbatim): the chunk-start state h_c (bf16 [K][V]), the record
// Bk | Qg | Khat | Aqk | A with 2^G_last, and X^T, D^T.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

constexpr uint32_t U_H = 0, U_XT = 32768, U_O = 49152;  // phase (c) use of the union
constexpr uint32_t TMEM_COLS = 256;  // [0,64) X'^T / O^T, [64,128) D^T, [128,256) Khat^T D

struct FwdArgs {
  __nv_bfloat16 *o;   // [B*T][HV][V] or null
  float *hT;          // [N][HV][K][V] or null
  int *err;           // device error flag (a bounded wait gave up)
};

template <bool kOut>
__global__ void __launch_bounds__(kThr, 1)
kda_fwd_tc_kernel(Problem P, Workspace W, FwdArgs args, const __grid_constant__ TmaMaps maps) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  float *vec = (float *)(sm + OFF_VEC);
  float *betab = (float *)(sm + OFF_BETA);
  uint64_t *bar = (uint64_t *)(sm + OFF_MISC);
  uint32_t *tslot = (uint32_t *)(sm + OFF_MISC + 8);
  uint64_t *bar_kqg = (uint64_t *)(sm + OFF_MISC + 16), *bar_v = (uint64_t *)(sm + OFF_MISC + 24);
  uint64_t *bar_o = (uint64_t *)(sm + OFF_MISC + 32);
  unsigned char *U = sm + OFF_U;

  const int n = blockIdx.x, j = blockIdx.y;
  const int HV = P.HV, h = j / (HV / P.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, vhalf = warp >> 2;
  const int cown = quarter * 32 + lane;  // key channel = TMEM lane of the state epilogues
  const int4 si = W.seq[n];

  if (tid == 0) {
    bar_init(bar, 1);
    bar_init(bar_kqg, 1);
    bar_init(bar_v, 1);
    bar_init(bar_o, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter
  uint32_t phase = 0, phase_o = 0, kq_par = 0, v_par = 0;
  KDA_PT_DECL;

  float hreg[64];  // h[cown][64 * vhalf + x]
  {
    const size_t base = (((size_t)n * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4) {
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (P.h0 != nullptr) t = *reinterpret_cast<const float4 *>(P.h0 + base + x);
      hreg[x] = t.x; hreg[x + 1] = t.y; hreg[x + 2] = t.z; hreg[x + 3] = t.w;
    }
  }

  if (si.w > 0) {
    const int2 ch0 = chunk_span(si, 0);
    if (tid == 0) {
      tma_kqg(maps, sbase, ch0.x, h, j, true, bar_kqg);
      mbar_expect_tx(bar_v, 16384u);
      tma_tile(sbase + OFF_VRAW, &maps.v, j, ch0.x, bar_v);
    }
    load_beta(P, betab, ch0.x, ch0.y, j);
    cp_commit();
  }

  for (int ci = 0; ci < si.w; ++ci) {
    const int cidx = si.z + ci;
    const int2 ch = chunk_span(si, ci);
    const int t0 = ch.x, len = ch.y;
    const size_t slot = (size_t)cidx * HV + j;
    const float *beta = betab + (ci & 1) * kC;
    cp_wait_all();  // beta
    if (!kOut && tid == 0) bulk_wait_read();  // the previous chunk's saved tiles have left shared memory
    bar_wait(bar_kqg, kq_par, args.err);
    kq_par ^= 1;
    if (len < kC) {  // rows past the sequence end hold other tokens: clear them
      zero_tail(sm + OFF_KRAW, len);
      zero_tail(sm + OFF_QRAW, len);
      fence_async_smem();
    }
    __syncthreads();
    KDA_PT(0);

    phase_a<true>(sm, len, beta);
    KDA_PT(2);
    if (ci + 1 < si.w) {  // staging k, q, g consumed: prefetch the next chunk's
      const int2 nx = chunk_span(si, ci + 1);
      if (tid == 0) tma_kqg(maps, sbase, nx.x, h, j, true, bar_kqg);
      load_beta(P, betab + ((ci + 1) & 1) * kC, nx.x, nx.y, j);
      cp_commit();
    }
    KDA_PT(3);
    phase_b<true>(sm, beta);
    if (!kOut && tid == 0) {  // Bk, Qg, Khat, Aqk, A tiles (adjacent, 64 KB) and 2^G_last
      unsigned char *dst = W.tc_tiles + slot * kTileRecord;
      bulk_store(dst, sbase + OFF_BK, 65536u);
      bulk_store(dst + 65536, smem_u32(vec + V_GAML * kD), 512u);
      bulk_commit();
    }

    // ---------------- (c) state chain on tcgen05 ----------------
    bar_wait(bar_v, v_par, args.err);
    v_par ^= 1;
    if (len < kC) zero_tail(sm + OFF_VRAW, len);  // (ordered before the MMAs by the barrier below)
    {
      unsigned char *H = U + U_H;  // h row-major [c][v], bf16
#pragma unroll
      for (int x8 = 0; x8 < 8; ++x8) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = hreg[8 * x8 + e];
        const uint4 u = pack8(t);
        *reinterpret_cast<uint4 *>(H + sw_chunk(cown, 8 * vhalf + x8, kD)) = u;
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(8);
    const uint32_t aH = sbase + OFF_U + U_H, aXT = sbase + OFF_U + U_XT;
    // D^T reuses the X^T tile, except in states mode, where X^T is still being saved
    const uint32_t aD = kOut ? aXT : sbase + OFF_U + U_O;
    unsigned char *Dt = kOut ? U + U_XT : U + U_O;
    if (!kOut && tid == 0) {  // h_c for the backward
      bulk_store(W.tc_hs + slot * kD * kD, aH, 32768u);
      bulk_commit();
    }
    if (tid == 0) {  // X'^T[v][r] = sum_c h[c][v] Bk[r][c]   (M=128 v, N=64 r, K=128 c)
      const uint32_t id = idesc(128, 64, 1, 0);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma(tmem, desc_mn(aH, s, 16384), desc_k16(sbase + OFF_BK, s, kC), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    KDA_PT(9);
    {  // X^T[v][r] = beta_r v[r][v] - X'^T[v][r]  -> bf16 tile [v][r]
      const int v = cown, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tq + (uint32_t)r0, d);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = r0 + q8 * 8 + e;
          const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_VRAW + sw_off(r, v, kC)));
          x[e] = beta[r] * vv - d[q8 * 8 + e];
        }
        *reinterpret_cast<uint4 *>(U + U_XT + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(10);
    if (!kOut && tid == 0) {  // X^T tile for the backward
      bulk_store(W.tc_xt + slot * 16384, aXT, 16384u);
      bulk_commit();
    }
    if (ci + 1 < si.w && tid == 0) {  // v of this chunk consumed
      const int2 nx = chunk_span(si, ci + 1);
      mbar_expect_tx(bar_v, 16384u);
      tma_tile(sbase + OFF_VRAW, &maps.v, j, nx.x, bar_v);
    }
    if (tid == 0) {  // D^T[v][r] = sum_i X^T[v][i] A[r][i]   (M=128 v, N=64 r, K=64 i)
      const uint32_t id = idesc(128, 64, 0, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s) mma(tmem + 64, desc_k16(aXT, s, kD), desc_k16(sbase + OFF_AM, s, kC), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    KDA_PT(11);
    {  // D^T -> bf16 tile [v][r]
      const int v = cown, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tq + 64u + (uint32_t)r0, d);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = d[q8 * 8 + e];
        *reinterpret_cast<uint4 *>(Dt + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(12);
    if (!kOut && tid == 0) {  // D^T tile for the backward
      bulk_store(W.tc_dt + slot * 16384, aD, 16384u);
      bulk_commit();
    }
    if (tid == 0) {
      // U[c][v] = sum_r Khat[r][c] D[r][v]   (M=128 c, N=128 v, K=64 r): the carried state first
      const uint32_t id3 = idesc(128, 128, 1, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_mn(sbase + OFF_KH, s, 8192), desc_k16(aD, s, kD), id3, s > 0);
      commit(bar);
      if (kOut) {  // O^T[v][r] = sum_c h[c][v] Qg[r][c] + sum_i D^T[v][i] Aqk[r][i], while the state updates
        const uint32_t id = idesc(128, 64, 1, 0), id2 = idesc(128, 64, 0, 0);
#pragma unroll
        for (int s = 0; s < 8; ++s) mma(tmem, desc_mn(aH, s, 16384), desc_k16(sbase + OFF_QG, s, kC), id, s > 0);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma(tmem, desc_k16(aD, s, kD), desc_k16(sbase + OFF_AQK, s, kC), id2, 1);
        commit(bar_o);
      }
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    KDA_PT(13);
    {
      const float gl = vec[V_GAML * kD + cown];
      float d[32];
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        tmem_ld32(tq + 128u + (uint32_t)(64 * vhalf + 32 * hx), d);
#pragma unroll
        for (int e = 0; e < 32; ++e) hreg[32 * hx + e] = fmaf(gl, hreg[32 * hx + e], d[e]);
      }
    }
    if (kOut) {  // O^T -> staging tile [r][v], then coalesced 16-byte stores
      bar_wait(bar_o, phase_o, args.err);
      phase_o ^= 1;
      fence_after();
      const int v = cown, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tq + (uint32_t)r0, d);
      __nv_bfloat16 *Ot = (__nv_bfloat16 *)(U + U_O);
#pragma unroll
      for (int e = 0; e < 32; ++e) Ot[(r0 + e) * kD + v] = __float2bfloat16_rn(d[e]);
    }
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(14);
    if (kOut) {
      const uint4 *Ot = (const uint4 *)(U + U_O);
      for (int it = tid; it < len * 16; it += kThr) {
        const int r = it >> 4, jj = it & 15;
        *reinterpret_cast<uint4 *>(args.o + ((size_t)(t0 + r) * HV + j) * kD + jj * 8) = Ot[r * 16 + jj];
      }
    }
    KDA_PT(15);
  }

  if (args.hT != nullptr) {
    float *dst = args.hT + (((size_t)n * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4)
      *reinterpret_cast<float4 *>(dst + x) = make_float4(hreg[x], hreg[x + 1], hreg[x + 2], hreg[x + 3]);
  }
  if (!kOut && tid == 0) bulk_wait_all();  // the saved tiles are in global memory before the CTA exits
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_free(tmem, TMEM_COLS);
  }
  KDA_PT_FLUSH;
}

}  // namespace

KDA_PT_EXPORT(kda_debug_fwd_phase_cycles)

cudaError_t tc_forward(const Problem &P, const Workspace &W, void *o, float *hT, bool states,
                       int *err, cudaStream_t s) {
  cudaError_t e = launch_chunk_map(P, W, s);
  if (e != cudaSuccess || P.N == 0) return e;
  FwdArgs a{(__nv_bfloat16 *)o, hT, err};
  TmaMaps maps;
  if ((e = make_tma_maps(P, P.v, nullptr, &maps)) != cudaSuccess) return e;
  const dim3 grid(P.N, P.HV);
  if (states) {
    e = cudaFuncSetAttribute(kda_fwd_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    KDA_LAUNCH("kda_fwd_tc_states", s, kda_fwd_tc_kernel<false><<<grid, kThr, SMEM_BYTES, s>>>(P, W, a, maps));
  } else {
    e = cudaFuncSetAttribute(kda_fwd_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    KDA_LAUNCH("kda_fwd_tc", s, kda_fwd_tc_kernel<true><<<grid, kThr, SMEM_BYTES, s>>>(P, W, a, maps));
  }
  return cudaGetLastError();
}

}  // namespace kda
