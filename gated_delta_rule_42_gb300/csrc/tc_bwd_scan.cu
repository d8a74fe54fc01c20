// Reverse state-gradient scan of the bf16 chunked KDA backward (K, V = 64 or 128).
//
// One CTA walks the chunks of one (sequence, value head) from last to first,
// holding dh' -- the gradient of the chunk-END state -- in fp32 registers
// (thread = key channel c, half the value columns), starting from dhT (or 0).
// Per chunk, with the chunk tiles Bk = beta k 2^G, Qg = q~ 2^G, Khat =
// k 2^(G_last - G), Aqk, A and 2^G_last from the per-chunk record (one bulk
// copy per chunk: the scan reads no q, k, g or beta), on tcgen05:
//   dD^T = dO^T Aqk + dh'^T Khat^T        dD = Aqk^T dO + Khat dh'   (deltas' gradient)
//   dX^T = dD^T A                         dX = A^T dD                (through A = (I+L)^-1)
//   dh  <- diag(2^G_last) dh' + Qg^T dO - Bk^T dX                    (gradient of the chunk-start state)
// The last line is the reverse recurrence of FLA's bwd_dhu ("[Fix] Use unit KDA
// gate scale when A_log is omitted", fla-org/flash-linear-attention PR #1294,
// commit log).  Every operand is read straight from row-major tiles through K-
// or MN-major descriptors, and the minus sign of Bk^T dX is the instruction's
// negate-B bit, so dD and dX exist in one layout only: the [64][V] operand tile
// the per-chunk gradient kernel reads.  The scan saves, per chunk, with bulk
// stores from shared memory: dh' (bf16 [K][V]) and dD, dX (bf16 [64][V]); at
// the start of the sequence it writes dh0 (fp32).
//
// Two CTAs share an SM (113 KB of shared memory and 256 tensor-memory columns
// each), so all chains of a training batch are resident at once.  Tiles are
// reused as soon as they die: Khat becomes dD, the dh' tile becomes dX.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

// Shared-memory map (offsets from the 1024-aligned base).
constexpr uint32_t S_REC = 0;      // record: Bk | Khat | A | Aqk | Qg (64 KB); Khat -> dD [64 r][128 v]
constexpr uint32_t S_DO = 65536;   // dO [64][128] bf16
constexpr uint32_t S_DH = 81920;   // dh' [K][V] bf16 (swizzled, 32 KB) -> dX [64 i][128 v]
constexpr uint32_t S_TILES = 114688;
// mbarriers (MMA +0, loads +8) and the tmem slot (+16): in the alignment slack
// below the base when it fits, else after the tiles
constexpr uint32_t S_SMALL = 32;
constexpr uint32_t S_SMEM = S_TILES + 1024;
static_assert(S_SMEM + 1024 <= 233472 / 2, "two CTAs per SM (228 KB, 1 KB reserved per CTA)");
constexpr uint32_t TMEM_COLS = 256;  // [0,64) dD^T, [64,128) dX^T, [128,256) dh update
constexpr uint32_t kNegB = 1u << 14;  // instruction descriptor: negate the B operand

__global__ void __launch_bounds__(kThr, 2)
kda_bwd_scan_tc_kernel(Problem P, Workspace W, const float *__restrict__ dhT, float *__restrict__ dh0, int *err,
                       const __grid_constant__ TmaMaps maps) {
  extern __shared__ unsigned char smraw[];
  const uint32_t raw = smem_u32(smraw);
  const uint32_t slack = ((raw + 1023u) & ~1023u) - raw;
  unsigned char *sm = smraw + slack;
  const uint32_t sbase = raw + slack;
  unsigned char *small = slack >= S_SMALL ? smraw : sm + S_TILES;
  uint64_t *bar = (uint64_t *)small, *bar_ld = (uint64_t *)(small + 8);
  uint32_t *tslot = (uint32_t *)(small + 16);

  const int n = blockIdx.x, j = blockIdx.y;
  const int HV = P.HV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, vhalf = warp >> 2;
  const int cown = quarter * 32 + lane;  // key channel (state) or value column (dD, dX): the TMEM lane
  const int r0 = 32 * vhalf;             // the token rows this thread's epilogues cover
  const int4 si = W.seq[n];

  if (tid == 0) {
    bar_init(bar, 1);
    bar_init(bar_ld, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);
  uint32_t phase = 0, ld_par = 0;

  float dreg[64];  // dh'[cown][64 * vhalf + x]; rows past K and columns past V (a 64-wide head) stay zero
  const bool hlive = cown < P.K && 64 * vhalf < P.V;
  {
    const size_t base = (((size_t)n * HV + j) * P.K + cown) * P.V + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4) {
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      if (dhT != nullptr && hlive) t = *reinterpret_cast<const float4 *>(dhT + base + x);
      dreg[x] = t.x; dreg[x + 1] = t.y; dreg[x + 2] = t.z; dreg[x + 3] = t.w;
    }
  }

  // one chunk's record (bulk copy) and dO rows (TMA), issued by one thread
  auto load_chunk = [&](int ci) {
    const int2 ch = chunk_span(si, ci);
    mbar_expect_tx(bar_ld, 65536u + 16384u);
    bulk_load(sbase + S_REC, W.tc_tiles + ((size_t)(si.z + ci) * HV + j) * kTileRecord, 65536u, bar_ld);
    tma_tile(sbase + S_DO, &maps.d, j, ch.x, bar_ld);
  };
  if (si.w > 0 && tid == 0) load_chunk(si.w - 1);

  for (int ci = si.w - 1; ci >= 0; --ci) {
    const int len = chunk_span(si, ci).y;
    const size_t slot = (size_t)(si.z + ci) * HV + j;
    // 2^G_last of this thread's key channel, read from the record in global memory
    const float gaml = reinterpret_cast<const float *>(W.tc_tiles + slot * kTileRecord + kRecGAML)[cown];
    {  // dh' -> bf16 operand tile, row-major [c][v]
      unsigned char *DH = sm + S_DH;
#pragma unroll
      for (int x8 = 0; x8 < 8; ++x8) {
        float t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = dreg[8 * x8 + e];
        *reinterpret_cast<uint4 *>(DH + sw_chunk(cown, 8 * vhalf + x8, kD)) = pack8(t);
      }
    }
    bar_wait(bar_ld, ld_par, err);
    ld_par ^= 1;
    if (len < kC) zero_tail(sm + S_DO, len);  // rows past the sequence end hold the next tokens
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {
      bulk_store(W.tc_dh + slot * kD * kD, sbase + S_DH, 32768u);  // dh' for the per-chunk kernel
      bulk_commit();
      // dD^T[v][r] = sum_i dO[i][v] Aqk[i][r] + sum_c dh'[c][v] Khat[r][c]   (M=128 v, N=64 r)
      const uint32_t id1 = idesc(128, 64, 1, 1), id2 = idesc(128, 64, 1, 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem, desc_mn(sbase + S_DO, s, 8192), desc_mn(sbase + S_REC + kRecAQK, s, 8192), id1, s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma(tmem, desc_mn(sbase + S_DH, s, 16384), desc_k16(sbase + S_REC + kRecKH, s, kC), id2, 1);
      commit(bar);
    }
    bar_wait(bar, phase, err);
    phase ^= 1;
    fence_after();
    {  // dD -> bf16 tile [r][v] in place of Khat (its product is complete)
      const int v = cown;
      float d[32];
      tmem_ld32(tq + (uint32_t)r0, d);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        *reinterpret_cast<__nv_bfloat16 *>(sm + S_REC + kRecKH + sw_off(r0 + e, v, kC)) = __float2bfloat16_rn(d[e]);
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {
      bulk_store(W.tc_dd + slot * kC * kD, sbase + S_REC + kRecKH, 16384u);  // dD for the per-chunk kernel
      bulk_commit();
      // dh' has left its tile before the product whose completion lets every
      // thread write dX there is issued; dD may still be in flight
      bulk_wait_read_all_but_one();
      // dX^T[v][i] = sum_r dD[r][v] A[r][i]   (M=128 v, N=64 i, K=64 r)
      const uint32_t id = idesc(128, 64, 1, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 64, desc_mn(sbase + S_REC + kRecKH, s, 8192), desc_mn(sbase + S_REC + kRecAM, s, 8192), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, err);
    phase ^= 1;
    fence_after();
    {  // dX -> bf16 tile [i][v] in place of dh'
      const int v = cown;
      float d[32];
      tmem_ld32(tq + 64u + (uint32_t)r0, d);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        *reinterpret_cast<__nv_bfloat16 *>(sm + S_DH + sw_off(r0 + e, v, kC)) = __float2bfloat16_rn(d[e]);
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {
      bulk_store(W.tc_dx + slot * kC * kD, sbase + S_DH, 16384u);  // dX for the per-chunk kernel
      bulk_commit();
      // U[c][v] = sum_r Qg[r][c] dO[r][v] - sum_r Bk[r][c] dX[r][v]   (M=128 c, N=128 v, K=64 r)
      const uint32_t id = idesc(128, 128, 1, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_mn(sbase + S_REC + kRecQG, s, 8192), desc_mn(sbase + S_DO, s, 8192), id, s > 0);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_mn(sbase + S_REC, s, 8192), desc_mn(sbase + S_DH, s, 8192), id | kNegB, 1);
      commit(bar);
    }
    bar_wait(bar, phase, err);
    phase ^= 1;
    fence_after();
    if (tid == 0) {
      bulk_wait_read();  // dD and dX have left shared memory
      if (ci > 0) load_chunk(ci - 1);  // every tile is dead: the previous chunk's loads go now
    }
    {  // dh <- diag(2^G_last) dh' + U
#pragma unroll
      for (int hx = 0; hx < 4; ++hx) {
        float d[16];
        tmem_ld16(tq + 128u + (uint32_t)(64 * vhalf + 16 * hx), d);
#pragma unroll
        for (int e = 0; e < 16; ++e) dreg[16 * hx + e] = fmaf(gaml, dreg[16 * hx + e], d[e]);
      }
    }
    fence_before();
    __syncthreads();  // the dX tile has been read: the dh' tile of the next step may overwrite it
    fence_after();
  }

  if (dh0 != nullptr && hlive) {
    float *dst = dh0 + (((size_t)n * HV + j) * P.K + cown) * P.V + 64 * vhalf;
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
  TmaMaps maps;
  cudaError_t e = make_tma_maps(P, P.v, dO, &maps);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kda_bwd_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  if (e != cudaSuccess) return e;
  KDA_LAUNCH("kda_bwd_scan_tc", s,
             kda_bwd_scan_tc_kernel<<<dim3(P.N, P.HV), kThr, S_SMEM, s>>>(P, W, dhT, dh0, err, maps));
  return cudaGetLastError();
}

}  // namespace kda
