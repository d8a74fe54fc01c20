// Sequential bf16 chunked KDA forward on the sm_103a tensor cores (K, V = 64 or 128).
//
// One CTA walks the chunks of one (sequence, value head) in order, keeping the
// fp32 state h[K][V] in registers (thread = key channel c, half the value
// columns).  The V-independent tiles of each chunk (Bk, Qg, Khat, Aqk, A and
// 2^G_last) come from the record the preparation kernel wrote (tc_prep.cu), by
// one bulk copy, so a chunk step is only the state chain on tcgen05 (operands
// in shared memory, fp32 accumulators in tensor memory):
//   X^T = (beta v)^T - h^T Bk^T          X = beta v - (beta k 2^G) h
//   D^T = X^T A^T                         D = u - w h, the chunk's deltas
//   O^T = h^T Qg^T + D^T Aqk^T            o = (q~ 2^G) h + Aqk D
//   h  <- diag(2^G_last) h + Khat^T D     the carried state
// h and Khat are stored row-major and read as MN-major operands, so no tile is
// ever transposed.  This is the state pass of the FLA KDA/GDN chunk pipeline
// (fwd_h + fwd_o, named in the commit log of "[Fix] Use unit KDA gate scale when
// A_log is omitted", fla-org/flash-linear-attention PR #1294) in one kernel,
// with the [K, V] fp32 state held on chip across chunks as in the recurrent_kda
// kernel of "kda in torchtitan (training)" (pytorch/torchtitan PR #4164).
//
// Two CTAs share an SM (113 KB of shared memory and 256 tensor-memory columns
// each), so all (sequence, head) chains of a training batch are resident at
// once and one CTA's loads and MMA round trips overlap the other's epilogues.
// The tiles are reused as soon as they die: v becomes X^T, Bk becomes D^T, the
// h tile becomes the output staging, and the next chunk's loads are issued as
// soon as the last products of this chunk complete.
//
// Four modes.  Output: o (and hT).  States (no output): the kernel saves, per
// chunk, what the backward needs beside the record -- the chunk-start state
// h_c (bf16 [K][V]) and X^T, D^T, as bulk copies of the swizzled tiles -- when
// the backward recomputes the forward.  Output + save: both at once, for a
// forward whose context the backward keeps.  Neither: the final state alone.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

// Shared-memory map (offsets from the 1024-aligned base).
constexpr uint32_t S_REC = 0;         // record: Bk | Khat | A | Aqk | Qg (64 KB; states mode: the first 40 KB); Bk -> D^T [128 v][64 r]
constexpr uint32_t S_V = 65536;       // v [64][128] bf16 -> X^T [128 v][64 r]
constexpr uint32_t S_H = 81920;       // h [K][V] bf16 (swizzled) -> output staging [64][128] bf16
constexpr uint32_t S_TILES = 114688;
// beta [64] fp32 (+0), mbarriers (MMA +256, loads +264, output MMA +272), tmem slot +280:
// in the alignment slack below the base when it fits, else after the tiles
constexpr uint32_t S_SMALL = 320;
constexpr uint32_t S_SMEM = S_TILES + 1024;
static_assert(S_SMEM + 1024 <= 233472 / 2, "two CTAs per SM (228 KB, 1 KB reserved per CTA)");
constexpr uint32_t TMEM_COLS = 256;  // [0,64) X'^T / O^T, [64,128) D^T, [128,256) Khat^T D


struct FwdArgs {
  __nv_bfloat16 *o;   // [B*T][HV][V] or null
  float *hT;          // [N][HV][K][V] or null
  int *err;           // device error flag (a bounded wait gave up)
};

template <int kMode>
__global__ void __launch_bounds__(kThr, 2)
kda_fwd_tc_kernel(Problem P, Workspace W, FwdArgs args, const __grid_constant__ TmaMaps maps) {
  extern __shared__ unsigned char smraw[];
  const uint32_t raw = smem_u32(smraw);
  const uint32_t slack = ((raw + 1023u) & ~1023u) - raw;
  unsigned char *sm = smraw + slack;
  const uint32_t sbase = raw + slack;
  unsigned char *small = slack >= S_SMALL ? smraw : sm + S_TILES;
  float *beta = (float *)small;
  uint64_t *bar = (uint64_t *)(small + 256), *bar_ld = (uint64_t *)(small + 264);
  uint64_t *bar_o = (uint64_t *)(small + 272);
  uint32_t *tslot = (uint32_t *)(small + 280);

  const int n = blockIdx.x, j = blockIdx.y;
  const int HV = P.HV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, vhalf = warp >> 2;
  const int cown = quarter * 32 + lane;  // key channel (state) or value column (X, D, O): the TMEM lane
  const int r0 = 32 * vhalf;             // the token columns this thread's epilogues cover
  const int4 si = W.seq[n];
  constexpr bool kOut = (kMode & kFwdOutput) != 0, kSave = (kMode & kFwdSave) != 0;
  constexpr uint32_t kRecBytes = kOut ? 65536u : kRecStates;  // the states pass needs Bk, Khat and A only

  if (tid == 0) {
    bar_init(bar, 1);
    bar_init(bar_ld, 1);
    bar_init(bar_o, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter
  uint32_t phase = 0, phase_o = 0, ld_par = 0;
  KDA_PT_DECL;

  float hreg[64];  // h[cown][64 * vhalf + x]; rows past K and columns past V (a 64-wide head) stay zero
  const bool hlive = cown < P.K && 64 * vhalf < P.V;
  {
    const size_t base = (((size_t)n * HV + j) * P.K + cown) * P.V + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4) {
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (P.h0 != nullptr && hlive) t = *reinterpret_cast<const float4 *>(P.h0 + base + x);
      hreg[x] = t.x; hreg[x + 1] = t.y; hreg[x + 2] = t.z; hreg[x + 3] = t.w;
    }
  }

  if (si.w > 0) {  // chunk 0: record and v (one thread, on bar_ld), beta (cp.async)
    const int2 ch0 = chunk_span(si, 0);
    if (tid == 0) {
      mbar_expect_tx(bar_ld, kRecBytes + 16384u);
      bulk_load(sbase + S_REC, W.tc_tiles + ((size_t)si.z * HV + j) * kTileRecord, kRecBytes, bar_ld);
      tma_tile(sbase + S_V, &maps.v, j, ch0.x, bar_ld);
    }
    load_beta(P, beta, ch0.x, ch0.y, j);
    cp_commit();
  }

  for (int ci = 0; ci < si.w; ++ci) {
    const int2 ch = chunk_span(si, ci);
    const int t0 = ch.x, len = ch.y;
    const size_t slot = (size_t)(si.z + ci) * HV + j;
    // 2^G_last of this thread's key channel, read from the record in global memory
    // (needed only at the state update, so the load latency hides behind the chain)
    const float gaml = reinterpret_cast<const float *>(W.tc_tiles + slot * kTileRecord + kRecGAML)[cown];
    {  // h -> bf16 operand tile, row-major [c][v]
      unsigned char *H = sm + S_H;
#pragma unroll
      for (int x8 = 0; x8 < 8; ++x8) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = hreg[8 * x8 + e];
        *reinterpret_cast<uint4 *>(H + sw_chunk(cown, 8 * vhalf + x8, kD)) = pack8(t);
      }
    }
    cp_wait_all();  // beta
    bar_wait(bar_ld, ld_par, args.err);
    ld_par ^= 1;
    if (len < kC) zero_tail(sm + S_V, len);  // rows past the sequence end hold the next tokens
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(0);
    if (kSave && tid == 0) {  // h_c for the backward
      bulk_store(W.tc_hs + slot * kD * kD, sbase + S_H, 32768u);
      bulk_commit();
    }
    if (tid == 0) {  // X'^T[v][r] = sum_c h[c][v] Bk[r][c]   (M=128 v, N=64 r, K=128 c)
      const uint32_t id = idesc(128, 64, 1, 0);
#pragma unroll
      for (int s = 0; s < 8; ++s) mma(tmem, desc_mn(sbase + S_H, s, 16384), desc_k16(sbase + S_REC, s, kC), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    KDA_PT(1);
    {  // X^T[v][r] = beta_r v[r][v] - X'^T[v][r] -> bf16 tile [v][r], in place of v
      const int v = cown;
      float d[32];
      tmem_ld32(tq + (uint32_t)r0, d);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int r = r0 + e;
        const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + S_V + sw_off(r, v, kC)));
        d[e] = beta[r] * vv - d[e];
      }
      __syncthreads();  // every thread has read its v values: the tile becomes X^T
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = d[q8 * 8 + e];
        *reinterpret_cast<uint4 *>(sm + S_V + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(2);
    if (kSave && tid == 0) {  // X^T tile for the backward
      bulk_store(W.tc_xt + slot * 16384, sbase + S_V, 16384u);
      bulk_commit();
    }
    if (tid == 0) {  // D^T[v][r] = sum_i X^T[v][i] A[r][i]   (M=128 v, N=64 r, K=64 i)
      const uint32_t id = idesc(128, 64, 0, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 64, desc_k16(sbase + S_V, s, kD), desc_k16(sbase + S_REC + kRecAM, s, kC), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    KDA_PT(3);
    {  // D^T -> bf16 tile [v][r] in place of Bk (its product is complete)
      const int v = cown;
      float d[32];
      tmem_ld32(tq + 64u + (uint32_t)r0, d);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = d[q8 * 8 + e];
        *reinterpret_cast<uint4 *>(sm + S_REC + sw_chunk(v, (r0 >> 3) + q8, kD)) = pack8(x);
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(4);
    if (kSave && tid == 0) {  // D^T tile for the backward
      bulk_store(W.tc_dt + slot * 16384, sbase + S_REC, 16384u);
      bulk_commit();
    }
    if (tid == 0) {
      // U[c][v] = sum_r Khat[r][c] D[r][v]   (M=128 c, N=128 v, K=64 r): the carried state first
      const uint32_t id3 = idesc(128, 128, 1, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_mn(sbase + S_REC + kRecKH, s, 8192), desc_k16(sbase + S_REC, s, kD), id3, s > 0);
      commit(bar);
      if (kOut) {  // O^T[v][r] = sum_c h[c][v] Qg[r][c] + sum_i D^T[v][i] Aqk[r][i], while the state updates
        const uint32_t id = idesc(128, 64, 1, 0), id2 = idesc(128, 64, 0, 0);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma(tmem, desc_mn(sbase + S_H, s, 16384), desc_k16(sbase + S_REC + kRecQG, s, kC), id, s > 0);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma(tmem, desc_k16(sbase + S_REC, s, kD), desc_k16(sbase + S_REC + kRecAQK, s, kC), id2, 1);
        commit(bar_o);
      }
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    if (kOut) {
      bar_wait(bar_o, phase_o, args.err);
      phase_o ^= 1;
    }
    fence_after();
    KDA_PT(5);
    // Every tile but h is dead: the next chunk's loads go now.
    if (kSave && tid == 0) bulk_wait_read();  // h_c, X^T, D^T have left shared memory
    if (ci + 1 < si.w) {
      const int2 nx = chunk_span(si, ci + 1);
      if (tid == 0) {
        mbar_expect_tx(bar_ld, kRecBytes + 16384u);
        bulk_load(sbase + S_REC, W.tc_tiles + (slot + HV) * kTileRecord, kRecBytes, bar_ld);
        tma_tile(sbase + S_V, &maps.v, j, nx.x, bar_ld);
      }
      load_beta(P, beta, nx.x, nx.y, j);
      cp_commit();
    }
    {  // h <- diag(2^G_last) h + U
#pragma unroll
      for (int hx = 0; hx < 4; ++hx) {
        float d[16];
        tmem_ld16(tq + 128u + (uint32_t)(64 * vhalf + 16 * hx), d);
#pragma unroll
        for (int e = 0; e < 16; ++e) hreg[16 * hx + e] = fmaf(gaml, hreg[16 * hx + e], d[e]);
      }
    }
    if (kOut) {  // O^T -> staging tile [r][v] over the h tile, then coalesced 16-byte stores
      if (kSave) __syncthreads();  // the h_c copy out of the h tile is complete
      const int v = cown;
      __nv_bfloat16 *Ot = (__nv_bfloat16 *)(sm + S_H);
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        float d[16];
        tmem_ld16(tq + (uint32_t)(r0 + 16 * hx), d);
#pragma unroll
        for (int e = 0; e < 16; ++e) Ot[(r0 + 16 * hx + e) * kD + v] = __float2bfloat16_rn(d[e]);
      }
      fence_before();
      __syncthreads();
      fence_after();
      const uint4 *Os = (const uint4 *)(sm + S_H);
      const int vq = P.V >> 3;  // 16-byte chunks of an output row (the padded columns are not stored)
      for (int it = tid; it < len * vq; it += kThr) {
        const int r = it / vq, jj = it - r * vq;
        *reinterpret_cast<uint4 *>(args.o + ((size_t)(t0 + r) * HV + j) * P.V + jj * 8) = Os[r * 16 + jj];
      }
    }
    fence_before();
    __syncthreads();  // the h tile (or the staging over it) is free for the next chunk
    fence_after();
    KDA_PT(6);
  }

  if (args.hT != nullptr && hlive) {
    float *dst = args.hT + (((size_t)n * HV + j) * P.K + cown) * P.V + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4)
      *reinterpret_cast<float4 *>(dst + x) = make_float4(hreg[x], hreg[x + 1], hreg[x + 2], hreg[x + 3]);
  }
  if (kSave && tid == 0) bulk_wait_all();  // the saved tiles are in global memory before the CTA exits
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

template <int kMode>
cudaError_t launch_fwd(const char *name, const Problem &P, const Workspace &W, const FwdArgs &a,
                       const TmaMaps &maps, cudaStream_t s) {
  cudaError_t e =
      cudaFuncSetAttribute(kda_fwd_tc_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  if (e != cudaSuccess) return e;
  KDA_LAUNCH(name, s, kda_fwd_tc_kernel<kMode><<<dim3(P.N, P.HV), kThr, S_SMEM, s>>>(P, W, a, maps));
  return cudaGetLastError();
}

cudaError_t tc_records(const Problem &P, const GateArgs &ga, const Workspace &W, int *err, cudaStream_t s) {
  cudaError_t e = launch_chunk_map(P, W, s);
  if (e != cudaSuccess || P.N == 0) return e;
  TmaMaps maps;
  if ((e = make_tma_maps(P, P.v, nullptr, &maps)) != cudaSuccess) return e;
  return tc_prepare(P, ga, W, maps, err, s);
}

cudaError_t tc_forward(const Problem &P, const GateArgs &ga, const Workspace &W, void *o, float *hT, int mode,
                       bool records_ready, int *err, cudaStream_t s) {
  cudaError_t e = records_ready ? launch_chunk_map(P, W, s) : tc_records(P, ga, W, err, s);
  if (e != cudaSuccess || P.N == 0) return e;
  FwdArgs a{(__nv_bfloat16 *)o, hT, err};
  TmaMaps maps;
  if ((e = make_tma_maps(P, P.v, nullptr, &maps)) != cudaSuccess) return e;
  switch (mode) {
    case 0: return launch_fwd<0>("kda_fwd_tc_final_state", P, W, a, maps, s);
    case kFwdOutput: return launch_fwd<kFwdOutput>("kda_fwd_tc", P, W, a, maps, s);
    case kFwdSave: return launch_fwd<kFwdSave>("kda_fwd_tc_states", P, W, a, maps, s);
    case kFwdOutput | kFwdSave: return launch_fwd<kFwdOutput | kFwdSave>("kda_fwd_tc_save", P, W, a, maps, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kda
