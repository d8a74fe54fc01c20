// Per-chunk gradients of the bf16 chunked KDA backward on one decay reference
// per chunk and channel: every contraction of the gradient chain is a plain
// tensor-core product.
//
// The pairwise decay 2^(G_r - G_i) of a chunk is split at the middle m of the
// channel's range over the chunk (m = (G_first + G_last) / 2):
//   row factor e1 = 2^(G_r - m),  column factor e2 = 2^(m - G_i),
// both within 2^(+-span/2).  With span = G_first - G_last <= kChunkSpan for
// every channel the decayed tiles Kr = k e1, Qr = q~ e1 and Kc = k e2 carry the
// whole chunk, and the chain
//   xr = tril_{-1}(dL) Kc,  yr = tril(dAqk) Kc,  xyi = X^T Kr + dAqk^T Qr
// is three 64-deep products with no per-block factor (the block-reference
// kernel in tc_bwd_intra.cu needs one per 16-token block pair).  A slot whose
// span is wider is listed (W.wide_cgrad, status word 5) for that kernel, whose
// results replace this launch's.
//
// Every product runs transposed, channel on the tensor-memory lane and token
// row on the column (M = 128, fp32 in TMEM):
//   [h dX^T | h dO^T][c][r] = [-dBk | dQg]      (one N = 128 product),
//   (dh' D^T)[c][r] = dKhat,
//   Z = [dO; dD][X; D]^T                        (N = 128: the dAqk and dA blocks),
//   [xr^T | yr^T] = Kc^T [dL; dAqk]^T            (one N = 128 product),
//   xyi^T = Kr^T X + Qr^T dAqk                  (hi/lo bf16 operands: three products per K step),
// so thread (warp w, lane l) owns channel c = 32 (w % 4) + l and the 16 rows of
// block w / 4, reads its values of every product with 32x32b tensor-memory
// loads, assembles on the packed fp32x2 pipe, two rows at a time (with
// Gamma = 2^G = e1 2^m, khat = 2^(G_last - G) = e2 2^(G_last - m))
//   dq~ = dQg Gamma + e1 yr
//   dk  = dKhat khat + beta Gamma dBk + beta e1 xr + e2 xyi
//   dG  = ln2 [dQg q~ Gamma + beta dBk k Gamma]                  (Q part)
//       + ln2 [beta k e1 xr + q~ e1 yr - k e2 xyi - dKhat k khat] (P part: sums to zero over the chunk
//                                                                   with the dG_last term)
//   dbeta = sum_v dX v + sum_c (dBk k Gamma + k e1 xr)
// and runs the reverse cumsum dg of its channel over its rows in registers, the
// block totals exchanged in shared memory.  Between the first products and the
// chain the CTA splits in two groups of 8 warps: one turns dA into T = A^T dA and
// dL = -tril_{-1}(T A^T) on warp MMAs while the other loads raw k and q, runs
// the gate's cumsum and builds the decayed tiles.  These are the intra-chunk backward
// steps of FLA's chunk_bwd_dqkwg / chunk_bwd_dv_local / prepare_wy_repr_bwd
// ("[Fix] Use unit KDA gate scale when A_log is omitted",
// fla-org/flash-linear-attention PR #1294, commit log); the inputs and their
// three prefetch groups are those of the block-reference kernel.  All
// reductions run in a fixed order: the result is bitwise reproducible.
#include "tc_intra.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;
using namespace intra;

// Widest per-channel decay span (log2) of a chunk that one middle reference
// carries (every factor within 2^(+-kChunkSpan / 2)).
constexpr float kChunkSpan = 192.f;
// Tensor memory columns (M = 128 accumulators: lane = channel, column = row).
constexpr uint32_t T_NBK = 0, T_DQG = 64, T_DKH = 128, T_Z = 192, T_XR = 320, T_YR = 384, T_XYI = 448;
static_assert(T_DQG == T_NBK + 64, "h [dX; dO]^T is one N = 128 product");
constexpr uint32_t TMEM_COLS = 512;
static_assert(T_YR == T_XR + 64, "xr and yr are one N = 128 product");
// Chain tiles of this kernel in [96 KB, 128 KB): dA [64 m][64 i] (then dL [64 r][64 i]) and
// dAqk [64 r][64 i] back to back, so [dL; dAqk] is one 128-row K-major operand; their lo
// twins 16 KB on.
constexpr uint32_t CK_DA = C_DAB, CK_DAQK = C_DAB + 8192;
static_assert(CK_DAQK + 8192 + LO128 <= C_XB, "dA/dL and dAqk with their lo twins");
// From the products to the chain the CTA runs as two groups of 8 warps (named barriers 1
// and 2): raw k and q land in the Kr hi and lo tiles' places, so the second group's tiles
// and the first group's dA, dAqk, T, dL and X tiles are disjoint.  A few loops of the two
// groups stay rolled ("#pragma unroll 1"): the kernel's code is large, and with the KDA
// gate's code inside it an unrolled version spent most of its stalls on instruction fetch.
constexpr int kGroupWarps = 8;
constexpr int kBarChainGroup = 1, kBarTileGroup = 2;
// Raw k and q land in the Kr hi and lo tiles' places once the products that read them (the
// dh' D^T and Z operands D^T and X^T) are done; the decayed-tile pass rewrites each 16-byte
// chunk in the thread that read it.
constexpr uint32_t CK_KRAW = C_KR, CK_QRAW = C_KR + LO128;
static_assert(CK_KRAW == I_XT && CK_QRAW == I_DT, "raw k, q over the X^T and D^T operands");
static_assert(C_KC + 2 * 16384 <= CK_DA && CK_DAQK + 8192 + LO128 <= C_XB && C_T + 16384 <= C_G,
              "the two groups' tiles are disjoint");
// Barrier among the 256 threads of one group.
__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(kGroupWarps * 32) : "memory");
}
// The same, returning whether any of the group's threads passed a nonzero v.
__device__ __forceinline__ bool group_sync_or(int id, int v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(v), "r"(id), "r"(kGroupWarps * 32)
      : "memory");
  return r != 0;
}
constexpr float kLn2 = 0.69314718055994530942f;
// The gate tile arrives by TMA with group P2: dense [64][128] fp32 rows (rows
// past the chunk hold other tokens until the cumsum overwrites them).
constexpr int kGD = kGT;
constexpr uint32_t kBytesG = kC * kD * 4u;
static_assert(kC * kGD * 4 <= C_A - C_G, "the dense gate tile fits the padded one's place");
// beta of a slot (cp.async from 64 threads; zero past len)
__device__ __forceinline__ void issue_beta(float *beta, const Problem &P, const Slot &q) {
  const int tid = threadIdx.x;
  if (tid < kC) {
    if (tid < q.len) cp4(smem_u32(beta + tid), P.beta + (size_t)(q.t0 + tid) * P.HV + q.j);
    else beta[tid] = 0.f;
  }
  cp_commit();
}
// Scalar gate (one decay per token and value head): the scalars of a slot's rows
// (zero past len), loaded into registers by every thread ...
constexpr int kSgIt = kC * 32 / kCT;  // float4 stores of the gate tile per thread
__device__ __forceinline__ void sg_load(float (&x)[kSgIt], const Problem &P, const Slot &q) {
#pragma unroll
  for (int u = 0; u < kSgIt; ++u) {
    const int r = (int)(threadIdx.x + u * kCT) >> 5;
    x[u] = r < q.len ? P.g[(size_t)(q.t0 + r) * P.HV + q.j] : 0.f;
  }
}
// ... and repeated over the 128 channels of the gate tile once the tile is free.
__device__ __forceinline__ void sg_store(float *G, const float (&x)[kSgIt]) {
#pragma unroll
  for (int u = 0; u < kSgIt; ++u) {
    const int it = threadIdx.x + u * kCT, r = it >> 5, c4 = (it & 31) * 4;
    *reinterpret_cast<float4 *>(G + r * kGD + c4) = make_float4(x[u], x[u], x[u], x[u]);
  }
}
// Rows of the vector table this kernel uses: G_last, 2^G_last, m, 2^m,
// 2^(G_last - m); the dg scan's block totals (Q, P, Khat term) x 4 blocks go to
// twelve rows it leaves free.
constexpr int V_M = V_RREF, V_EM = V_EREF, V_LM = V_LAM;
constexpr int V_SG = V_RREF + 1;  // kSG: dg row sums [4 channel quarters][64 rows] (two vector rows)
// kL2 (the fused L2-norm backward): the rows' inverse norms (k rows 0..63, q rows 64..127)
// in a vector row, and the row dots y . dy of q and of k as [64 rows][4 channel quarters]
// tables in the KDA gate's partials area (written there only after the dg scan)
constexpr int V_RN = V_RREF + 3;
static_assert(V_RN < V_EREF, "a free vector row");
constexpr uint32_t C_DOTQ = C_GPB, C_DOTK = C_GPB + 1024;
static_assert(C_DOTK + 1024 <= C_GPA, "the dot tables fit the partials area");
// Sum of v[t] over the warp's 32 lanes for each of 4 rows t: on return lanes 8t .. 8t + 7
// hold row t's sum.
__device__ __forceinline__ float rows4_sum(float (&v)[4]) {
  const int lane = threadIdx.x & 31;
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool up = (lane & 8) != 0;
    const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float t = v[0];
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}
// kL2: four values per row parked in tensor memory, in the columns of this thread's lane the
// assembly has just read (T_NBK, T_DQG, T_DKH, T_XR + row): each (lane, column) belongs to
// one thread, which reads it back after the CTA barrier.  Four consecutive rows at a time.
__device__ __forceinline__ void tmem_park4x4(uint32_t t, const float (&a)[4], const float (&b)[4],
                                             const float (&c)[4], const float (&d)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%4,%5,%6,%7};\n"
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%1], {%8,%9,%10,%11};\n"
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%2], {%12,%13,%14,%15};\n"
      "tcgen05.st.sync.aligned.32x32b.x4.b32 [%3], {%16,%17,%18,%19};\n" ::"r"(t + T_NBK),
      "r"(t + T_DQG), "r"(t + T_DKH), "r"(t + T_XR), "r"(__float_as_uint(a[0])), "r"(__float_as_uint(a[1])),
      "r"(__float_as_uint(a[2])), "r"(__float_as_uint(a[3])), "r"(__float_as_uint(b[0])), "r"(__float_as_uint(b[1])),
      "r"(__float_as_uint(b[2])), "r"(__float_as_uint(b[3])), "r"(__float_as_uint(c[0])), "r"(__float_as_uint(c[1])),
      "r"(__float_as_uint(c[2])), "r"(__float_as_uint(c[3])), "r"(__float_as_uint(d[0])), "r"(__float_as_uint(d[1])),
      "r"(__float_as_uint(d[2])), "r"(__float_as_uint(d[3]))
      : "memory");
}
__device__ __forceinline__ void tmem_unpark4x4(uint32_t t, float (&a)[4], float (&b)[4], float (&c)[4], float (&d)[4]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%16];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%17];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%18];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12,%13,%14,%15}, [%19];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(t + T_NBK), "r"(t + T_DQG), "r"(t + T_DKH), "r"(t + T_XR)
      : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[4 + i]);
    c[i] = __uint_as_float(r[8 + i]);
    d[i] = __uint_as_float(r[12 + i]);
  }
}
// (dg/dx, dg/dA_log) of the KDA gate at x on the hardware exponential, logarithm and
// reciprocal (bf16-path accuracy).  The unbounded form g = -s softplus(x) takes both from
// one exponential e = exp(-|x|): sigmoid(x) = (x >= 0 ? 1 : e) / (1 + e) and
// softplus(x) = max(x, 0) + ln(1 + e); the bounded form g = lb sigmoid(s x) as before.
__device__ __forceinline__ float2 gate_grad(float x, float s, float lb) {
  if (lb < 0.f) return kgate_grad_fast(x, s, lb);
  const float e = __expf(-fabsf(x)), r = __fdividef(1.f, 1.f + e);
  const float sg = x >= 0.f ? r : e * r, sp = fmaxf(x, 0.f) + __logf(1.f + e);
  return make_float2(-s * sg, -s * sp);
}
__device__ __forceinline__ int tot_row(int kind, int R) {
  const int k = 4 * kind + R;
  return k < 6 ? V_D + k : V_LAM + 2 + (k - 6);
}

// Four consecutive columns of six accumulators for this thread's lane, then
// one wait (the registers are tied to the wait so nothing reads them early).
__device__ __forceinline__ void tmem_ld6x4(uint32_t t, float (&a)[4], float (&b)[4], float (&c)[4], float (&d)[4],
                                           float (&e)[4], float (&f)[4]) {
  uint32_t r[24];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%24];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%25];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%26];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12,%13,%14,%15}, [%27];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%16,%17,%18,%19}, [%28];\n"
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%20,%21,%22,%23}, [%29];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
      : "r"(t + T_NBK), "r"(t + T_DQG), "r"(t + T_DKH), "r"(t + T_XR), "r"(t + T_YR), "r"(t + T_XYI)
      : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[4 + i]);
    c[i] = __uint_as_float(r[8 + i]);
    d[i] = __uint_as_float(r[12 + i]);
    e[i] = __uint_as_float(r[16 + i]);
    f[i] = __uint_as_float(r[20 + i]);
  }
}
// The bf16 at byte offset off of a tile, as fp32.
__device__ __forceinline__ float bf_at(const unsigned char *tile, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + off));
}
// Sum of v[t] over the warp's 32 lanes for each of 16 rows t: on return lanes
// 2t and 2t + 1 hold row t's sum in v[0] (a butterfly that halves the rows it
// carries at each step: 16 shuffles).
__device__ __forceinline__ float rows16_sum(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int w = 8, o = 16; w >= 1; w >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w], keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// kGate: the KDA gate inside the op; kSG: one decay per (token, value head), dg summed over
// the channels (the two are not combined); kL2: the q/k L2-norm prologue with HV = H, its
// backward dx = r (dy - y (y . dy)) fused: a first pass over the assembly parks each
// element's dy and y in tensor-memory columns it has read and forms the row dots, a second
// pass after a barrier (and after the next slot's last loads are issued) stores dq, dk.
template <bool kGate, bool kSG, bool kL2>
__global__ void __launch_bounds__(kCT, 1)
kda_bwd_intra_chunk_tc_kernel(Problem P, Workspace W, IntraArgs args, const __grid_constant__ TmaMaps maps,
                              GateArgs ga) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int HV = P.HV, H = P.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;
  float *G = (float *)(sm + C_G);
  float *vec = (float *)(sm + C_VEC);
  float *beta = (float *)(sm + C_BETA);
  float *rb = (float *)(sm + C_RB);
  float *red = (float *)(sm + C_RED);  // [0, 64): sum_v dX v; [64, 192): d(2^G_last)
  uint64_t *bar_s = (uint64_t *)(sm + C_MISC), *bar_p1 = bar_s + 1, *bar_p2 = bar_s + 2;
  uint64_t *bar_kq = bar_s + 3, *bar = bar_s + 4, *bar_g = bar_s + 6;  // (bar_s + 5 holds the tmem slot)
  uint32_t *tslot = (uint32_t *)(sm + C_MISC + 40);
  const float qscale = head_qscale(P.K);  // 1/sqrt(K)
  KDA_PT_DECL;

  if (tid == 0) {
    for (int b = 0; b < 5; ++b) bar_init(bar_s + b, 1);
    bar_init(bar_g, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter

  int64_t s_idx = blockIdx.x;
  Slot cur, nxt;  // this slot and the next (its chunk-table entry loaded an iteration ahead)
  bool have = get_slot<kAllSlots>(P, W, s_idx, 0, cur);
  bool more = get_slot<kAllSlots>(P, W, s_idx + gridDim.x, 0, nxt);
  if (have) {  // the first slot: every group at once
    if (tid == 0) {
      mbar_expect_tx(bar_s, kBytesS);
      mbar_expect_tx(bar_p1, kBytesP1);
      mbar_expect_tx(bar_p2, kBytesP2 + (kSG ? 0u : kBytesG));
      for (int i = 0; i < kCopiesS; ++i) copy_s(i, sbase, W, maps, cur, bar_s);
      for (int i = 0; i < kCopiesP1; ++i) copy_p1(i, sbase, W, maps, cur, bar_p1);
      for (int i = 0; i < kCopiesP2; ++i) copy_p2(i, sbase, W, maps, cur, bar_p2);
      if (!kSG) tma_load3(sbase + C_G, &maps.g, 0, cur.j, cur.t0, bar_p2);
    }
    if (kSG) {
      float x[kSgIt];
      sg_load(x, P, cur);
      sg_store(G, x);
    }
    issue_beta(beta, P, cur);
  }
  for (uint32_t it = 0; have; ++it) {
    const uint32_t par = it & 1u;
    const int t0 = cur.t0, len = cur.len, j = cur.j, h = cur.h;
    // the chunk-table entry of the slot after next: loaded now, decoded at the end of the
    // slot (nothing waits for the load in between)
    const int64_t s_n2 = s_idx + 2 * (int64_t)gridDim.x;
    const bool in_n2 = s_n2 < (int64_t)P.NC * HV;
    const int c_n2 = in_n2 ? (int)(s_n2 / HV) : 0;
    const int4 ent_n2 = W.chunk[c_n2];
    bool ok = true;  // every bounded wait of this thread succeeded
    float gsc = 0.f, gbias = 0.f;  // kGate: the slot's gate scale and the bias of channel tid % 128
    if (kGate) {  // (loaded here: the gate pass and the dg scan use them thousands of cycles on)
      gsc = kgate_scale(ga, j);
      gbias = (tid & 127) < P.K ? kgate_bias(ga, P.K, j, tid & 127) : 0.f;
    }
    KDA_PT(13);
    ok &= bar_wait(bar_s, par, args.err);
    ok &= bar_wait(bar_p1, par, args.err);
    ok &= bar_wait(bar_p2, par, args.err);
    if (len < kC)  // dO rows past the sequence end hold other tokens: clear them
      for (int it2 = tid; it2 < (kC - len) * 16; it2 += kCT) {
        const int r = 64 + len + (it2 >> 4), q = it2 & 15;
        *reinterpret_cast<uint4 *>(sm + I_STK + sw_chunk(r, q, 192)) = make_uint4(0, 0, 0, 0);
      }
    cp_wait_all();  // beta
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(14);

    // ---- tensor-core products, transposed (M = 128 channels or rows of [X; D]) ----
    if (tid == 0) {
      const uint32_t idk = idesc(128, 128, 0, 0), idd = idesc(128, 64, 0, 1), idz = idesc(128, 128, 0, 1);
      // (dh' D^T)[c][r] = sum_v dh'[c][v] D[r][v]   (D^T is stored [v][r]: an MN-major B)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + T_DKH, desc_k16(sbase + I_DH, k, kD), desc_mn(sbase + I_DT, k, 8192), idd, k > 0);
      // Z[n'][i'] = sum_v [dO; dD][n'][v] [X; D][i'][v]   ([X; D]^T is stored [v][i']: an MN-major B)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + T_Z, desc_k16(sbase + I_STK + 64 * 128, k, 192), desc_mn(sbase + I_XT, k, 16384), idz, k > 0);
      commit(bar_g);  // X^T and D^T are read: raw k, q may land there
      // [(h dX^T) | (h dO^T)][c][n] = sum_v h[c][v] [dX; dO][n][v]   (K = 128 v; T_DQG = T_NBK + 64)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + T_NBK, desc_k16(sbase + I_H, k, kD), desc_k16(sbase + I_STK, k, 192), idk, k > 0);
      commit(bar);
      if (bar_wait(bar_g, par, args.err)) {  // raw k, q
        fence_async_smem();
        mbar_expect_tx(bar_kq, 32768u);
        tma_tile(sbase + CK_KRAW, &maps.k, h, t0, bar_kq);
        tma_tile(sbase + CK_QRAW, &maps.q, h, t0, bar_kq);
      } else {
        ok = false;
      }
    }
    // meanwhile (warp 0 only issues the products): warps 4..7 d(2^G_last)[c] =
    // sum_v dh'[c][v] h[c][v]; warps 1..3, 8..15 dv = beta dX and sum_v dX v
    if (warp >= 4 && warp < 8) {
      const int c = tid - kD;
      float acc = 0.f;
#pragma unroll 4
      for (int jj = 0; jj < 16; ++jj) {
        float a[8], b[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + I_H + sw_chunk(c, jj, kD)), a);
        unpack8(*reinterpret_cast<const uint4 *>(sm + I_DH + sw_chunk(c, jj, kD)), b);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(a[e], b[e], acc);
      }
      red[64 + c] = acc;
    }
    const int rw = warp < 4 ? warp - 1 : warp - 5;  // 0..10 on warps 1..3 and 8..15
    for (int r = rw; warp != 0 && (warp < 4 || warp >= 8) && r < kC; r += 11) {  // one warp per row
      float part = 0.f;
      if (r < len) {
        const float br = beta[r];
        const int v0 = lane * 4;
        const uint2 xd = *reinterpret_cast<const uint2 *>(sm + I_STK + sw_off(r, v0, 192));
        const uint2 xv = *reinterpret_cast<const uint2 *>(sm + I_V + sw_off(r, v0, kC));
        const float2 d01 = unpack_bf16(xd.x), d23 = unpack_bf16(xd.y);
        const float2 v01 = unpack_bf16(xv.x), v23 = unpack_bf16(xv.y);
        if (v0 < P.V)  // (a 64-wide head: the padded columns are not stored)
          *reinterpret_cast<uint2 *>(args.dv + ((size_t)(t0 + r) * HV + j) * P.V + v0) =
              make_uint2(pack_bf16(br * d01.x, br * d01.y), pack_bf16(br * d23.x, br * d23.y));
        part = d01.x * v01.x + d01.y * v01.y + d23.x * v23.x + d23.y * v23.y;
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      }
      if (lane == 0) red[r] = part;
    }
    KDA_PT(15);
    ok &= bar_wait(bar, 0u, args.err);  // (two commits per slot: products, then the chain)
    fence_after();
    __syncthreads();  // products in TMEM; the operand tiles are dead
    KDA_PT(0);

    // ---- two warp groups until the chain: warps 0..7 take dA and dAqk out of TMEM and run
    // T = A^T dA and dL; warps 8..15 load the raw k, q rows and build G, the reference and the
    // decayed tiles.  Their tiles are disjoint: the raw rows land in the Kr hi and lo tiles'
    // places (dead product operands), each 16-byte chunk rewritten by the thread that read it. ----
    if (kGate) {  // the decay from the raw gate, on every warp before the groups part: channel
                  // tid % 128, rows tid / 128 + 4 i
      const int cg = tid & 127;
      if (cg < P.K) {
#pragma unroll
        for (int i = 0; i < kC / 4; ++i) {
          const int r = (tid >> 7) + 4 * i;
          if (r < len) G[r * kGD + cg] = kgate_fast(G[r * kGD + cg] + gbias, gsc, ga.lb);
        }
      }
      __syncthreads();
    }
    if (warp < kGroupWarps) {
      {  // Z: lanes 0..63 (r), cols 64..127 (i) = dAqk[r][i]; lanes 64..127 (m), cols 0..63 (i) = dA[m][i]
        const int ch = warp >> 2, row = 32 * (quarter & 1) + lane;  // ch: the column half
        const bool qk = quarter < 2;
        float x[32];
        tmem_ld32(tq + T_Z + (qk ? 64u : 0u) + (uint32_t)(32 * ch), x);
#pragma unroll
        for (int hx = 0; hx < 4; ++hx) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int col = 32 * ch + 8 * hx + e;
            y[e] = (qk && col > row) ? 0.f : x[8 * hx + e];  // dAqk[r][i] is a gradient of Aqk only where i <= r
          }
          uint4 hi, lo;
          split8(y, hi, lo);
          const uint32_t off = sw_chunk(row, 4 * ch + hx, kC);
          *reinterpret_cast<uint4 *>(sm + (qk ? CK_DAQK : CK_DA) + off) = hi;
          *reinterpret_cast<uint4 *>(sm + (qk ? CK_DAQK : CK_DA) + LO128 + off) = lo;
        }
      }
      group_sync(kBarChainGroup);
      KDA_PT(1);
      // ---- T = A^T dA  (T[r][m] = sum_i' A[i'][r] dA[i'][m]); a warp: 16 rows, 32 columns ----
      const int mt = warp >> 1, nh = warp & 1;
      {
        float acc[4][4] = {};
#pragma unroll 1
        for (int s = 0; s < 4; ++s) {
          uint32_t a[4];
          lda_t(sbase + C_A, kC, 16 * mt, 16 * s, a);  // element (r, i') = A[i'][r]
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            uint32_t bh[4], bl[4];
            ldb_t(sbase + CK_DA, kC, 32 * nh + 16 * qq, 16 * s, bh);  // element (i', m) = dA[i'][m]
            ldb_t(sbase + CK_DA + LO128, kC, 32 * nh + 16 * qq, 16 * s, bl);
            mma16816(acc[2 * qq], a, bh[0], bh[1]);
            mma16816(acc[2 * qq], a, bl[0], bl[1]);
            mma16816(acc[2 * qq + 1], a, bh[2], bh[3]);
            mma16816(acc[2 * qq + 1], a, bl[2], bl[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * mt + (lane >> 2) + 8 * hh, m = 32 * nh + 8 * nt + (lane & 3) * 2;
            st_split2(sm + C_T, LO64, r, m, kC, acc[nt][2 * hh], acc[nt][2 * hh + 1]);
          }
      }
      group_sync(kBarChainGroup);  // (every read of dA has ended: its tiles become dL)
      KDA_PT(3);
      // ---- dL = -tril_{-1}(T A^T); X = beta dL.  A warp: the 16-column blocks nh and nh + 2
      // of its 16 rows; the blocks above the diagonal are zero (no product, zeros stored). ----
#pragma unroll 1
      for (int qq = 0; qq < 2; ++qq) {
        const int nq = nh + 2 * qq;
        float acc[2][4] = {};
        if (nq <= mt) {
#pragma unroll 1
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
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * mt + (lane >> 2) + 8 * hh, i = 16 * nq + 8 * nt + (lane & 3) * 2;
            const float d0 = (i < r) ? -acc[nt][2 * hh] : 0.f, d1 = (i + 1 < r) ? -acc[nt][2 * hh + 1] : 0.f;
            st_split2(sm + CK_DA, LO128, r, i, kC, d0, d1);
            st_split2(sm + C_XB, LO64, r, i, kC, beta[r] * d0, beta[r] * d1);
          }
      }
      KDA_PT(22);
    } else {
      const int tb = tid - kGroupWarps * 32;  // 0..255
      int wide_c = 0;
      if (tb < kD) {  // G and the reference m = (G_first + G_last) / 2 per channel
        const int c = tb;
        float s = 0.f;
        float col[kC];
#pragma unroll
        for (int r = 0; r < kC; ++r) col[r] = G[r * kGD + c];
#pragma unroll
        for (int r = 0; r < kC; ++r) {
          if (r < len) s += col[r];
          col[r] = s;
        }
#pragma unroll
        for (int r = 0; r < kC; ++r) G[r * kGD + c] = col[r];
        const float gl = s, m = 0.5f * (col[0] + gl);  // rows past len hold G_last
        wide_c = !(col[0] - gl <= kChunkSpan);        // (NaN-safe)
        vec[V_GL * kD + c] = gl;
        vec[V_GAML * kD + c] = exp2f(gl);
        vec[V_M * kD + c] = m;
        vec[V_EM * kD + c] = exp2f(m);
        vec[V_LM * kD + c] = exp2f(gl - m);
      }
      KDA_PT(19);
      ok &= bar_wait(bar_kq, par, args.err);  // raw k, q
      KDA_PT(20);
      if (len < kC)  // rows past the sequence end hold other tokens: clear them
        for (int it2 = tb; it2 < (kC - len) * 16; it2 += kGroupWarps * 32) {
          const int r = len + (it2 >> 4), q = it2 & 15;
          const uint32_t off = (q >> 3) * 8192 + r * 128 + (q & 7) * 16;
          *reinterpret_cast<uint4 *>(sm + CK_KRAW + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(sm + CK_QRAW + off) = make_uint4(0, 0, 0, 0);
        }
      // a channel's decay span is wider than one reference carries: list the slot for the
      // block-reference kernel (whose results replace this launch's)
      if (group_sync_or(kBarTileGroup, wide_c) && tb == 0) W.wide_cgrad[atomicAdd(W.flags + 5, 1)] = (int)cur.slot;
      KDA_PT(21);
      {  // the decayed hi/lo tiles Kr = k e1, Qr = q~ e1, Kc = k e2; a half-warp per row
        const int jj = tb & 15, c0 = jj * 8, rg = tb >> 4;  // four rows per thread
        float mv[8];
#pragma unroll
        for (int e = 0; e < 8; e += 4)
          *reinterpret_cast<float4 *>(mv + e) = *reinterpret_cast<const float4 *>(vec + V_M * kD + c0 + e);
#pragma unroll 1
        for (int rr = 0; rr < 4; ++rr) {  // (rolled: the kernel's code stays within the instruction cache)
          const int r = rg * 4 + rr;
          const uint32_t off = sw_chunk(r, jj, kC);
          float kv[8], qv[8], o[8], e1[8], e2[8];
          unpack8(*reinterpret_cast<const uint4 *>(sm + CK_KRAW + off), kv);  // raw k, q (zero past len)
          unpack8(*reinterpret_cast<const uint4 *>(sm + CK_QRAW + off), qv);
          if (P.l2norm) {  // q/k L2-norm prologue (value-head partials: its backward runs per q/k head afterwards)
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              sk = fmaf(kv[e], kv[e], sk);
              sq = fmaf(qv[e], qv[e], sq);
            }
#pragma unroll
            for (int o2 = 1; o2 < 16; o2 <<= 1) {
              sk += __shfl_xor_sync(0xffffffffu, sk, o2);
              sq += __shfl_xor_sync(0xffffffffu, sq, o2);
            }
            const float rk = 1.0f / sqrtf(sk + kL2NormEps), rq = 1.0f / sqrtf(sq + kL2NormEps);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              kv[e] *= rk;
              qv[e] *= rq;
            }
            if (kL2 && jj == 0) {  // the rows' inverse norms, for the fused backward
              vec[V_RN * kD + r] = rk;
              vec[V_RN * kD + kC + r] = rq;
            }
          }
          float g[8];  // (two 16-byte reads: a half-warp reads one whole row, free of bank conflicts)
          *reinterpret_cast<float4 *>(g) = *reinterpret_cast<const float4 *>(G + r * kGD + c0);
          *reinterpret_cast<float4 *>(g + 4) = *reinterpret_cast<const float4 *>(G + r * kGD + c0 + 4);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            e1[e] = ex2(g[e] - mv[e]);  // within 2^(+-kChunkSpan/2)
            e2[e] = ex2(mv[e] - g[e]);
          }
          uint4 hi, lo;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = kv[e] * e1[e];
          split8(o, hi, lo);
          *reinterpret_cast<uint4 *>(sm + C_KR + off) = hi;          // (over the raw k chunk read above)
          *reinterpret_cast<uint4 *>(sm + C_KR + LO128 + off) = lo;  // (over the raw q chunk read above)
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
      KDA_PT(23);
    }
    fence_async_smem();  // Kr, Qr, Kc, dAqk, dL and X are read by the tensor core next
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(4);
    // ---- the chain, from one thread (a commit tracks the products its own thread issued) ----
    if (tid == 96) {
      const uint32_t id_yi = idesc(128, 64, 1, 1), id_xyr = idesc(128, 128, 1, 0), id_xi = idesc(128, 64, 1, 1);
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int p = 0; p < 3; ++p) {  // hi*hi, hi*lo, lo*hi
          const uint32_t la = p == 2 ? LO128 : 0u, lb = p == 1 ? LO128 : 0u;
          // yi^T[c][i] = sum_r Qr[r][c] dAqk[r][i]        (A: Qr MN-major; B: dAqk MN-major)
          mma(tmem + T_XYI, desc_mn(sbase + C_QR + la, s, 8192), desc_mn(sbase + CK_DAQK + lb, s, 8192), id_yi,
              (s > 0 || p > 0) ? 1u : 0u);
        }
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int p = 0; p < 3; ++p) {
          const uint32_t la = p == 2 ? LO128 : 0u;
          // [xr^T | yr^T][c][n] = sum_i Kc[i][c] [dL; dAqk][n][i]   (B: [dL; dAqk] K-major, 128 rows)
          mma(tmem + T_XR, desc_mn(sbase + C_KC + la, s, 8192), desc_k16(sbase + CK_DA + (p == 1 ? LO128 : 0u), s, kC),
              id_xyr, (s > 0 || p > 0) ? 1u : 0u);
          // xi^T[c][i] = sum_r Kr[r][c] X[r][i], onto yi   (B: X MN-major)
          mma(tmem + T_XYI, desc_mn(sbase + C_KR + la, s, 8192), desc_mn(sbase + C_XB + (p == 1 ? LO64 : 0u), s, 8192),
              id_xi, 1u);
        }
      commit(bar);
    }
    ok &= bar_wait(bar, 1u, args.err);
    fence_after();
    KDA_PT(5);
    if (more) {  // the next slot's dh', v, A and h columns 64..127 into the dead dAqk^T, X, T, A and dL tiles
      if (tid == 0) mbar_expect_tx(bar_p1, kBytesP1);
      if (lane == 0 && warp >= 1 && warp <= kCopiesP1) {
        fence_async_smem();
        copy_p1(warp - 1, sbase, W, maps, nxt, bar_p1);
      }
    }

    // ---- assembly: thread = (channel c, rows 16 R .. 16 R + 15), rows in pairs on the packed
    // fp32x2 pipe; k e2 = (k e1) e2 e2 (k e1 e2 is k itself: no overflow) ----
    const int c = 32 * quarter + lane, R = warp >> 2;
    const float gm = vec[V_M * kD + c], em = vec[V_EM * kD + c], lm = vec[V_LM * kD + c];
    const float2 ngm = make_float2(-gm, -gm), em2 = make_float2(em, em), lm2 = make_float2(lm, lm);
    const float2 ln2 = make_float2(kLn2, kLn2), eln2 = make_float2(kLn2 * em, kLn2 * em);
    float qv[16], pv[16], bp[16];  // dG's Q and P parts, dbeta partials of the 16 rows
    float cq = 0.f;                // sum over the rows of dKhat k khat
    const bool cin = c < P.K;      // (a 64-wide head: the padded channels are not stored)
    const bool odd = (lane & 1) != 0;
    const int cp = c & ~1;         // the channel pair a store covers
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
      float tb[4], tg[4], th[4], tx[4], ty[4], tz[4];  // -dBk, dQg, dKhat, xr, yr, xyi
      tmem_ld6x4(tq + (uint32_t)(16 * R + 4 * s4), tb, tg, th, tx, ty, tz);
      if (s4 == 1) KDA_PT(18);
      const float4 b4 = *reinterpret_cast<const float4 *>(beta + 16 * R + 4 * s4);
      float dq4[4], dk4[4];  // kL2: y . dy of the quad's rows over this thread's channel
      float pdq[4], pyq[4], pyk[4], pdk[4];  // kL2: dy and y of the quad's rows, parked below
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const int t = 4 * s4 + u, r = 16 * R + t;  // rows r, r + 1
        const uint32_t o0 = sw_off(r, c, kC), o1 = sw_off(r + 1, c, kC);
        const float2 Kr = __fadd2_rn(make_float2(bf_at(sm + C_KR, o0), bf_at(sm + C_KR, o1)),
                                     make_float2(bf_at(sm + C_KR + LO128, o0), bf_at(sm + C_KR + LO128, o1)));
        const float2 Qr = __fadd2_rn(make_float2(bf_at(sm + C_QR, o0), bf_at(sm + C_QR, o1)),
                                     make_float2(bf_at(sm + C_QR + LO128, o0), bf_at(sm + C_QR + LO128, o1)));
        const float2 d = __fadd2_rn(make_float2(G[r * kGD + c], G[(r + 1) * kGD + c]), ngm);  // G - m
        const float2 e1 = make_float2(ex2(d.x), ex2(d.y)), e2 = make_float2(ex2(-d.x), ex2(-d.y));
        const float2 Kc = __fmul2_rn(__fmul2_rn(Kr, e2), e2);
        const float2 br = u == 0 ? make_float2(b4.x, b4.y) : make_float2(b4.z, b4.w);
        const float2 dBk = make_float2(-tb[u], -tb[u + 1]), dQg = make_float2(tg[u], tg[u + 1]);
        const float2 dKh = make_float2(th[u], th[u + 1]), xr = make_float2(tx[u], tx[u + 1]);
        const float2 yr = make_float2(ty[u], ty[u + 1]), xyi = make_float2(tz[u], tz[u + 1]);
        const float2 gam = __fmul2_rn(e1, em2);
        const float2 dq2 = __ffma2_rn(dQg, gam, __fmul2_rn(e1, yr));
        float2 dk2 = __fmul2_rn(dKh, __fmul2_rn(e2, lm2));
        dk2 = __ffma2_rn(__fmul2_rn(br, gam), dBk, dk2);
        dk2 = __ffma2_rn(__fmul2_rn(br, e1), xr, dk2);
        dk2 = __ffma2_rn(e2, xyi, dk2);
        const float2 kht = __fmul2_rn(__fmul2_rn(dKh, Kc), lm2);  // dKhat k khat
        const float2 bdk = __fmul2_rn(br, dBk);
        const float2 qp = __fmul2_rn(eln2, __ffma2_rn(dQg, Qr, __fmul2_rn(bdk, Kr)));
        float2 pp = __fmul2_rn(__fmul2_rn(br, Kr), xr);
        pp = __ffma2_rn(Qr, yr, pp);
        pp = __ffma2_rn(make_float2(-Kc.x, -Kc.y), xyi, pp);
        pp = __fmul2_rn(ln2, __fadd2_rn(pp, make_float2(-kht.x, -kht.y)));
        const float2 bq = __ffma2_rn(__fmul2_rn(dBk, Kr), em2, __fmul2_rn(Kr, xr));
        const bool in0 = r < len, in1 = r + 1 < len;
        qv[t] = in0 ? qp.x : 0.f;
        qv[t + 1] = in1 ? qp.y : 0.f;
        pv[t] = in0 ? pp.x : 0.f;
        pv[t + 1] = in1 ? pp.y : 0.f;
        cq += (in0 ? kht.x : 0.f) + (in1 ? kht.y : 0.f);
        bp[t] = bq.x;
        bp[t + 1] = bq.y;
        if (kL2) {  // first pass: park dy (dq2, dk2) and y (Qr e2 = q~ normalised, Kr e2 = k normalised)
          const float2 yq = __fmul2_rn(Qr, e2), yk = __fmul2_rn(Kr, e2);
          pdq[u] = dq2.x;
          pdq[u + 1] = dq2.y;
          pyq[u] = yq.x;
          pyq[u + 1] = yq.y;
          pyk[u] = yk.x;
          pyk[u + 1] = yk.y;
          pdk[u] = dk2.x;
          pdk[u + 1] = dk2.y;
          dq4[u] = yq.x * dq2.x;
          dq4[u + 1] = yq.y * dq2.y;
          dk4[u] = yk.x * dk2.x;
          dk4[u + 1] = yk.y * dk2.y;
        } else {  // lanes (c, c + 1) trade one value: the even lane stores row r, the odd lane row r + 1,
           // each as the channel pair (c & ~1, c | 1)
          const float gq = __shfl_xor_sync(0xffffffffu, odd ? dq2.x : dq2.y, 1);
          const float gk = __shfl_xor_sync(0xffffffffu, odd ? dk2.x : dk2.y, 1);
          const float2 pq = odd ? make_float2(gq, dq2.y) : make_float2(dq2.x, gq);
          const float2 pk = odd ? make_float2(gk, dk2.y) : make_float2(dk2.x, gk);
          if ((odd ? in1 : in0) && cin) {
            const size_t tok = (size_t)(t0 + r + (odd ? 1 : 0));
            if (args.partial) {  // (scaled in the group reduction)
              *reinterpret_cast<float2 *>((float *)args.dq + (tok * HV + j) * P.K + cp) = pq;
              *reinterpret_cast<float2 *>((float *)args.dk + (tok * HV + j) * P.K + cp) = pk;
            } else {
              *reinterpret_cast<uint32_t *>((__nv_bfloat16 *)args.dq + (tok * H + h) * P.K + cp) =
                  pack_bf16(pq.x * qscale, pq.y * qscale);
              *reinterpret_cast<uint32_t *>((__nv_bfloat16 *)args.dk + (tok * H + h) * P.K + cp) = pack_bf16(pk.x, pk.y);
            }
          }
        }
      }
      if (kL2) {  // the quad's row dots over the warp's 32 channels, into [row][quarter] tables
        tmem_park4x4(tq + (uint32_t)(16 * R + 4 * s4), pdq, pyq, pyk, pdk);
        const float tqd = rows4_sum(dq4), tkd = rows4_sum(dk4);
        if ((lane & 7) == 0) {
          const int row = 16 * R + 4 * s4 + (lane >> 3);
          reinterpret_cast<float *>(sm + C_DOTQ)[row * 4 + quarter] = tqd;
          reinterpret_cast<float *>(sm + C_DOTK)[row * 4 + quarter] = tkd;
        }
      }
    }
    float ar[16];  // kGate: the raw gate of this thread's rows, for the dg scan (loaded before it)
    if (kGate) {
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int r = 16 * R + t;
        ar[t] = (r < len && cin) ? __ldg(P.g + ((size_t)(t0 + r) * HV + j) * P.K + c) : 0.f;
      }
    }
    KDA_PT(9);
    // block totals of the dg scan: Q, P and the Khat term of rows 16 R ..
    {
      float tq_ = 0.f, tp_ = 0.f;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        tq_ += qv[t];
        tp_ += pv[t];
      }
      vec[tot_row(0, R) * kD + c] = tq_;
      vec[tot_row(1, R) * kD + c] = tp_;
      vec[tot_row(2, R) * kD + c] = cq;
    }
    // dbeta partials: the sum over this warp's 32 channels of each of its 16 rows
    {
      const float v = rows16_sum(bp);
      if ((lane & 1) == 0) rb[quarter * kC + 16 * R + (lane >> 1)] = v;
    }
    if (kL2) asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
    fence_before();
    // every read of the tiles, G and beta is done; the totals are published; every wait of
    // the slot is behind, so its outcome is known here (the KDA gate and the scalar gate
    // reduce theirs at the end of the slot, where their sums need a barrier anyway)
    bool all_ok = __syncthreads_and(ok) != 0;
    KDA_PT(10);
    if (more) {  // the next slot's remaining inputs into the dead tiles; its G and beta
      if (tid == 0) {
        mbar_expect_tx(bar_p2, kBytesP2 + (kSG ? 0u : kBytesG));
        mbar_expect_tx(bar_s, kBytesS);
      }
      if (lane == 0 && warp >= 1 && warp <= kCopiesP2 + kCopiesS + (kSG ? 0 : 1)) {
        fence_async_smem();
        if (warp <= kCopiesP2) copy_p2(warp - 1, sbase, W, maps, nxt, bar_p2);
        else if (warp <= kCopiesP2 + kCopiesS) copy_s(warp - 1 - kCopiesP2, sbase, W, maps, nxt, bar_s);
        else tma_load3(sbase + C_G, &maps.g, 0, nxt.j, nxt.t0, bar_p2);
      }
      issue_beta(beta, P, nxt);
    }
    if (kL2) {  // second pass: dq, dk = r (dy - y (y . dy)) from the parked values and the row dots
      fence_after();
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        float pdq[4], pyq[4], pyk[4], pdk[4];
        tmem_unpark4x4(tq + (uint32_t)(16 * R + 4 * q4), pdq, pyq, pyk, pdk);
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
          const int r = 16 * R + 4 * q4 + u;
          const float4 dqa = *reinterpret_cast<const float4 *>(sm + C_DOTQ + r * 16);
          const float4 dqb = *reinterpret_cast<const float4 *>(sm + C_DOTQ + (r + 1) * 16);
          const float4 dka = *reinterpret_cast<const float4 *>(sm + C_DOTK + r * 16);
          const float4 dkb = *reinterpret_cast<const float4 *>(sm + C_DOTK + (r + 1) * 16);
          const float2 dotq = make_float2(dqa.x + dqa.y + dqa.z + dqa.w, dqb.x + dqb.y + dqb.z + dqb.w);
          const float2 dotk = make_float2(dka.x + dka.y + dka.z + dka.w, dkb.x + dkb.y + dkb.z + dkb.w);
          const float2 rk = make_float2(vec[V_RN * kD + r], vec[V_RN * kD + r + 1]);
          const float2 rq = make_float2(vec[V_RN * kD + kC + r], vec[V_RN * kD + kC + r + 1]);
          const float2 dq2 = make_float2(pdq[u], pdq[u + 1]), yq = make_float2(pyq[u], pyq[u + 1]);
          const float2 yk = make_float2(pyk[u], pyk[u + 1]), dk2 = make_float2(pdk[u], pdk[u + 1]);
          // dq = rq (qscale dq2 - (yq / qscale) (y . dy)), dk = rk (dk2 - yk (y . dy)) (yq carries qscale)
          const float iqs = 1.f / qscale;
          const float2 fq = make_float2(rq.x * (qscale * dq2.x - yq.x * iqs * dotq.x),
                                        rq.y * (qscale * dq2.y - yq.y * iqs * dotq.y));
          const float2 fk = make_float2(rk.x * (dk2.x - yk.x * dotk.x), rk.y * (dk2.y - yk.y * dotk.y));
          const float gq = __shfl_xor_sync(0xffffffffu, odd ? fq.x : fq.y, 1);
          const float gk = __shfl_xor_sync(0xffffffffu, odd ? fk.x : fk.y, 1);
          const float2 pq = odd ? make_float2(gq, fq.y) : make_float2(fq.x, gq);
          const float2 pk = odd ? make_float2(gk, fk.y) : make_float2(fk.x, gk);
          if (r + (odd ? 1 : 0) < len && cin) {
            const size_t tok = (size_t)(t0 + r + (odd ? 1 : 0));
            *reinterpret_cast<uint32_t *>((__nv_bfloat16 *)args.dq + (tok * H + h) * P.K + cp) =
                pack_bf16(pq.x, pq.y);
            *reinterpret_cast<uint32_t *>((__nv_bfloat16 *)args.dk + (tok * H + h) * P.K + cp) = pack_bf16(pk.x, pk.y);
          }
        }
      }
      // (the KDA gate's partials go where the dot tables are, after the dg scan)
      if (kGate) __syncthreads();
    }
    float sgx[kSgIt];  // kSG: the next slot's scalars, stored into the gate tile at the end of the slot
    if (kSG && more) sg_load(sgx, P, nxt);
    float gpb = 0.f, gpa = 0.f;  // kGate: this thread's dbias and dA_log partials
    {  // dg = reverse cumsum of dG over the chunk (G in log2 units)
      float qoff = 0.f, poff = 0.f, ppre = 0.f, ks = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float tQ = vec[tot_row(0, b) * kD + c], tP = vec[tot_row(1, b) * kD + c];
        ks += vec[tot_row(2, b) * kD + c];
        if (b > R) {
          qoff += tQ;
          poff += tP;
        }
        if (b < R) ppre += tP;
      }
      // dg_t = sum_{s>=t} dG_s: the Q part and the carried-state decay term from
      // the chunk end; the zero-sum P part from whichever end is nearer
      // (sum_{s>=t} P_s = -sum_{s<t} P_s, the Khat column sum counted at the last
      // row), halving the cancelling terms it sums.
      KDA_PT(16);
      const int mid = len >> 1;
#pragma unroll
      for (int t = 0; t < 16; ++t) {  // rows before mid: the prefix, in place of the P part
        if (16 * R + t < mid) {
          const float x = pv[t];
          pv[t] = -ppre;
          ppre += x;
        }
      }
      KDA_PT(17);
      const float carried = kLn2 * vec[V_GAML * kD + c] * red[64 + c];
      float qs = qoff, ps = poff + kLn2 * ks;
      const float sc = gsc, gb = cin ? gbias : 0.f;  // (c == tid % 128: the channel whose bias it loaded)
      float sgr[16];  // kSG: this thread's dg of each row, summed over the channels below
#pragma unroll
      for (int p2 = 7; p2 >= 0; --p2) {
        float vv[2];
#pragma unroll
        for (int w = 1; w >= 0; --w) {
          const int t = 2 * p2 + w, r = 16 * R + t;
          const bool hi = r >= mid;
          qs += qv[t];
          if (hi) ps += pv[t];
          float v = qs + carried + (hi ? ps : pv[t]);
          if (kGate) {  // da = dG dg/da; the parameter gradients' partials
            const float2 d = gate_grad(ar[t] + gb, sc, ga.lb);
            const bool use = r < len && cin;
            gpb += use ? v * d.x : 0.f;
            gpa = use ? fmaf(v, d.y, gpa) : gpa;
            v *= d.x;
          }
          vv[w] = v;
          if (kSG) sgr[t] = (r < len && cin) ? v : 0.f;
        }
        if (!kSG) {  // lanes (c, c + 1) trade one value and store rows 2 p2 (even lane), 2 p2 + 1 (odd lane)
          const float got = __shfl_xor_sync(0xffffffffu, odd ? vv[0] : vv[1], 1);
          const int rs = 16 * R + 2 * p2 + (odd ? 1 : 0);
          if (rs < len && cin)
            *reinterpret_cast<float2 *>(args.dg + ((size_t)(t0 + rs) * HV + j) * P.K + cp) =
                odd ? make_float2(got, vv[1]) : make_float2(vv[0], got);
        }
      }
      if (kSG) {  // the sum over the warp's 32 channels of each row, then over the 4 quarters below
        const float v = rows16_sum(sgr);
        if ((lane & 1) == 0) vec[V_SG * kD + quarter * kC + 16 * R + (lane >> 1)] = v;
      }
    }
    KDA_PT(12);
    if (kGate) {
      reinterpret_cast<float *>(sm + C_GPB)[R * kD + c] = gpb;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gpa += __shfl_xor_sync(0xffffffffu, gpa, o);
      if (lane == 0) reinterpret_cast<float *>(sm + C_GPA)[warp] = gpa;
    }
    if (kGate || kSG) all_ok = __syncthreads_and(ok) != 0;
    KDA_PT(7);
    if (kGate) {  // the slot's partials, summed in a fixed order: dbias per channel, dA_log per slot
      if (tid < kD) {
        const float *gp = reinterpret_cast<const float *>(sm + C_GPB);
        W.gpart_b[cur.slot * kD + tid] = gp[tid] + gp[kD + tid] + gp[2 * kD + tid] + gp[3 * kD + tid];
      } else if (warp == kD / 32) {  // the 16 warp sums
        float t = lane < kCT / 32 ? reinterpret_cast<const float *>(sm + C_GPA)[lane] : 0.f;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) W.gpart_a[cur.slot] = t;
      }
    }
    if (tid < kC && tid < len)
      args.dbeta[(size_t)(t0 + tid) * HV + j] = red[tid] + rb[tid] + rb[kC + tid] + rb[2 * kC + tid] + rb[3 * kC + tid];
    if (kSG) {
      if (tid < kC && tid < len) {
        const float *sp = vec + V_SG * kD;
        args.dg[(size_t)(t0 + tid) * HV + j] = sp[tid] + sp[kC + tid] + sp[2 * kC + tid] + sp[3 * kC + tid];
      }
      if (more) sg_store(G, sgx);  // (the gate tile is dead; the loop top publishes it)
    }
    KDA_PT(8);
    if (!all_ok) {  // a wait gave up (error flag set): let the copies already issued land, then stop
      if (more) {
        if (tid == 0) {
          bar_wait(bar_s, par ^ 1u, args.err);
          bar_wait(bar_p1, par ^ 1u, args.err);
          bar_wait(bar_p2, par ^ 1u, args.err);
        }
        cp_wait_all();
      }
      break;
    }
    cur = nxt;
    have = more;
    nxt.j = (int)(s_n2 - (int64_t)c_n2 * HV);
    nxt.h = nxt.j / (HV / H);
    nxt.t0 = ent_n2.y;
    nxt.len = ent_n2.z;
    nxt.slot = (size_t)s_n2;
    more = in_n2 && ent_n2.x >= 0;
    s_idx += gridDim.x;
  }  // slot loop
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_free(tmem, TMEM_COLS);
  }
  KDA_PT_FLUSH;
}

}  // namespace

KDA_PT_EXPORT(kda_debug_intra_chunk_phase_cycles)

template <bool kGate, bool kSG, bool kL2>
cudaError_t launch_chunk(const Problem &P, const GateArgs &ga, const Workspace &W, const IntraArgs &a,
                         const TmaMaps &maps, unsigned grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_intra_chunk_tc_kernel<kGate, kSG, kL2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  KDA_LAUNCH("kda_bwd_intra_tc", s,
             kda_bwd_intra_chunk_tc_kernel<kGate, kSG, kL2><<<grid, kCT, C_SMEM, s>>>(P, W, a, maps, ga));
  return cudaGetLastError();
}

template <bool kL2>
cudaError_t launch_chunk_l2(const Problem &P, const GateArgs &ga, const Workspace &W, const IntraArgs &a,
                            const TmaMaps &maps, unsigned grid, cudaStream_t s) {
  if (P.scalar_gate) return launch_chunk<false, true, kL2>(P, ga, W, a, maps, grid, s);
  return ga.on ? launch_chunk<true, false, kL2>(P, ga, W, a, maps, grid, s)
               : launch_chunk<false, false, kL2>(P, ga, W, a, maps, grid, s);
}

cudaError_t launch_intra_chunk(const Problem &P, const GateArgs &ga, const Workspace &W, const IntraArgs &a,
                               const TmaMaps &maps, unsigned grid, cudaStream_t s) {
  // the L2-norm backward is fused when the q/k head's gradients come from one value head
  return (P.l2norm && !a.partial) ? launch_chunk_l2<true>(P, ga, W, a, maps, grid, s)
                                  : launch_chunk_l2<false>(P, ga, W, a, maps, grid, s);
}

}  // namespace kda
