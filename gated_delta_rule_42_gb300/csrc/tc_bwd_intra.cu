// Per-chunk gradients of the bf16 chunked KDA backward on 16-token block
// references: the tensor-core products and the gradient chain in one kernel.
// It runs over the slots the chunk-reference kernel (tc_bwd_chunk.cu) lists,
// those whose chunk decay span is too wide for one reference per chunk, and its
// fix-up launch over the slots with a 16-token block too wide for it in turn.
// (K, V = 64 run in the 128-wide tiles, zero-padded.)
//
// Persistent: one CTA (16 warps) per SM walks its slots,
// and loads the next slot's inputs into tiles as soon as the current slot's
// work leaves them dead (three groups, below), so most of each slot's loads
// overlap the previous slot's chain and assembly.  Inputs: the
// chunk-start state h and the tiles X^T (X = beta v - Bk h), D^T (D = A X) and
// A that the forward kept (or its recompute saved), the gradient of the
// chunk-end state dh', and dD, dX from the reverse scan.  First, on tcgen05
// (fp32 in TMEM):
//   dX h^T -> -dBk,  dO h^T -> dQg                             (two M=64 products)
//   dKhat = D dh'^T                                            (Khat = k 2^(G_last - G))
//   [X; D] [dO; dD]^T -> block (X, dD) = dA^T, block (D, dO) = dAqk^T
// and on the SIMT cores dv = beta dX, sum_v dX v and d(2^G_last) = rowsum(dh' .* h).
// The products never leave the chip: the chain reads them from TMEM.  It
// finishes
//   dL   = -tril_{-1}(A^T dA A^T)                 gradient through A = (I + L)^-1
//   the chain through L = beta*KK and Aqk to the keys, queries and gate,
// and assembles dq, dk, dg and dbeta.  With 2^(G_r - G_i) split per channel
// at 16-token block references exactly as in the record kernel (rows:
// e1 = 2^(G_r - Gr(R)), columns: e2 = 2^(Gc(I) - G_i), between blocks the
// factor D_RI = 2^(Gr(R) - Gc(I)) <= 1 on the block product; Gr = Gc = the
// middle of the block's range, or for a channel whose span exceeds kSpanMax
// the block's first and last row):
//   row side    xr = sum_i dL_ri  Kc_i D_RI,  yr = sum_i dAqk_ri Kc_i D_RI
//   column side xi = sum_r X_ri   Kr_r D_RI,  yi = sum_r dAqk_ri Qr_r D_RI   (X = beta dL)
// on 16x16 warp MMAs.  References in the middle of each block's range (Gr =
// Gc) keep every factor within 2^(+-kSpanMax/2); a slot with a block whose
// span is wider is listed for the fix-up launch of this kernel, which takes
// each block's first row as Gr and its last as Gc (factors <= 1), forms the
// diagonal blocks from the raw rows with pairwise exponents and carries true
// values (e1 = e2 = 1) into the assembly: exact for any gate.  Then per
// element (Gamma = 2^G, khat = 2^(G_last - G)):
//   dq~ = dQg Gamma + e1 yr
//   dk  = dKhat khat + beta Gamma dBk + beta e1 xr + e2 (xi + yi)
//   dG  = ln2 [dQg q~ Gamma - dKhat k khat + beta dBk k Gamma + beta k e1 xr + q~ e1 yr - k e2 (xi + yi)]
//   dG_last += ln2 (sum_r dKhat k khat + 2^G_last d(2^G_last))
//   dbeta   = sum_v dX v + sum_c (dBk k Gamma + k e1 xr)
//   dg = reverse cumsum of dG inside the chunk (G is in log2 units).
// These are the intra-chunk backward steps of FLA's chunk_bwd_dqkwg /
// chunk_bwd_dv_local / prepare_wy_repr_bwd ("[Fix] Use unit KDA gate scale when
// A_log is omitted", fla-org/flash-linear-attention PR #1294, commit log).
// All reductions run in a fixed order: the result is bitwise reproducible.
#include "tc_intra.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;
using namespace intra;

// Widest per-channel decay span (log2) of a 16-token block that the middle
// references carry (e1, e2 within 2^(+-kSpanMax / 2)); a slot with a wider
// block goes to the fix-up launch.
constexpr float kSpanMax = 192.f;
// Tensor memory: the per-chunk products that the assembly reads element-wise are
// M = 64 accumulators, whose 16-row block R sits in lanes 0..15 of lane quarter R:
// a warp of quarter R reads its 16 x 8 blocks straight in mma C-fragment order
// (tcgen05.ld .16x256b).  Z (M = 128) feeds the dA split only.
constexpr uint32_t TMEM_COLS = 512;   // [0,128) dX h^T, [128,256) dO h^T, [256,384) dKhat, [384,512) Z
// Assembly scratch in the dead dL .. T tiles: the segment and block totals of the
// final dg column scan.  dG itself is parked in the Kr / Qr tiles: once a thread
// has read its Kr, Qr (hi and lo) at (r, c..c+1), the 8 bytes of each pair slot
// hold dG's Q and P parts of (r, c) and (r, c+1).
// The assembly's Khat column terms [4 blocks][128] go to the vector rows of the
// block factors D_RI (dead after the pairwise chains), and the dg scan's segment
// totals (of Q for segments 1..7 -- segment 0's is never read -- and of P for
// segments 0..7) to 15 vector rows the scan does not read, so every chain tile
// is free for the next slot's inputs as soon as its own work ends.
constexpr float kLn2 = 0.69314718055994530942f;

// Element (a, b) of a hi/lo tile pair (64 columns, the lo twin LO64 bytes on).
__device__ __forceinline__ float hilo(const unsigned char *tile, int a, int b) {
  const uint32_t off = sw_off(a, b, kC);
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + off)) +
         __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + LO64 + off));
}
// Channels (c, c + 1) of row t of the chunk: k, or q~ = q / sqrt(K) (is_q), as the
// chain sees them (L2-normalised with the prologue, by the inverse norms in rb);
// zero past the chunk's length is the caller's guard.  For the exact path only.
__device__ __forceinline__ float2 raw_row(const Problem &P, const IntraArgs &a, int t0, int h, int t, int c,
                                          const float *rb, bool is_q) {
  (void)a;
  if (c >= P.K) return make_float2(0.f, 0.f);  // channels past a 64-wide head
  const __nv_bfloat16 *base = (const __nv_bfloat16 *)(is_q ? P.q : P.k);
  const float2 x = unpack_bf16(__ldg(reinterpret_cast<const unsigned int *>(base + ((size_t)(t0 + t) * P.H + h) * P.K + c)));
  float s = is_q ? head_qscale(P.K) : 1.f;
  if (P.l2norm) s *= rb[(is_q ? kC : 0) + t];
  return make_float2(x.x * s, x.y * s);
}

template <bool B>
struct BoolC {
  static constexpr bool value = B;
};
// Per-element operands of the gradient assembly.  Block-factor path: the decay
// tiles Kr = k e1, Qr = q~ e1, Kc = k e2, the vectors eref = 2^Gr, lam =
// 2^(G_last - Gc), and e1 = 2^(G - Gr), e2 = 2^(Gc - G), einv = 1 / e1 (kInv),
// with gm = Gr, ge = Gc.  Exact path: k, q~ themselves with e1 = e2 = einv = 1,
// eref = 2^G and lam = 2^(G_last - G), so that every product below means the
// same in both.
struct Opnd {
  float Kr, Qr, Kc, e1, e2, einv, eref, lam;
};
template <bool kWide, bool kInv>
__device__ __forceinline__ Opnd opnd(float Kr, float Qr, float Kc, float g, float gm, float ge, float eref, float lam,
                                     float kraw, float qraw) {
  Opnd o;
  if (kWide) {
    o.Kr = kraw; o.Qr = qraw; o.Kc = kraw;
    o.e1 = 1.f; o.e2 = 1.f; o.einv = 1.f;
    o.eref = ex2(g);
    o.lam = lam * ex2(ge - g);
  } else {
    o.Kr = Kr; o.Qr = Qr; o.Kc = Kc;
    o.e1 = ex2(g - gm);
    o.e2 = ex2(ge - g);
    o.einv = kInv ? ex2(gm - g) : 0.f;
    o.eref = eref;
    o.lam = lam;
  }
  return o;
}

// kScalarGate: g and dg are [tokens][HV] (one decay per token, repeated over the channels here).
// kL2: the q/k L2-norm prologue with HV = H, its backward fused: dx = r (dy - y (y . dy)) per
// (token, head) row, from the inverse norms r of the decay-tile pass and row dots y . dy that a
// first pass over the assembly's formulas forms, so dq and dk leave as bf16 in one pass.
// kSrc: the slots walked -- all, those the chunk-reference kernel left (chunk span too
// wide for it), or (the fix-up, kFix) those a block-reference launch listed for the exact path.
// kGate: the KDA gate inside the op (g holds the raw gate a): the cumsum makes the decay, and
// the dg scan writes da = dG dg/da and per-slot partials of dbias and dA_log (W.gpart_*).
template <bool kScalarGate, bool kL2, int kSrc, bool kGate>
__global__ void __launch_bounds__(kCT, 1)
kda_bwd_intra_tc_kernel(Problem P, Workspace W, IntraArgs args, const __grid_constant__ TmaMaps maps, GateArgs ga) {
  constexpr bool kFix = kSrc == kFixList;
  const int nlist = slot_list_count<kSrc>(W);
  if (kSrc != kAllSlots && (int)blockIdx.x >= nlist) return;
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
  uint64_t *bar_kq = bar_s + 3, *bar = bar_s + 4;
  uint32_t *tslot = (uint32_t *)(sm + C_MISC + 40);
  const float qscale = head_qscale(P.K);  // 1/sqrt(K)
  KDA_PT_DECL;

  if (tid == 0) {
    for (int b = 0; b < 5; ++b) bar_init(bar_s + b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter

  int64_t s_idx = blockIdx.x;
  Slot cur;
  bool have = get_slot<kSrc>(P, W, s_idx, nlist, cur);
  if (have) {  // the first slot: every group at once
    if (tid == 0) {
      mbar_expect_tx(bar_s, kBytesS);
      mbar_expect_tx(bar_p1, kBytesP1);
      mbar_expect_tx(bar_p2, kBytesP2);
      for (int i = 0; i < kCopiesS; ++i) copy_s(i, sbase, W, maps, cur, bar_s);
      for (int i = 0; i < kCopiesP1; ++i) copy_p1(i, sbase, W, maps, cur, bar_p1);
      for (int i = 0; i < kCopiesP2; ++i) copy_p2(i, sbase, W, maps, cur, bar_p2);
    }
    issue_gate_beta<kScalarGate>(sbase, sm, P, beta, cur);
  }
  for (uint32_t it = 0; have; ++it) {
    const uint32_t par = it & 1u;
    const int t0 = cur.t0, len = cur.len, j = cur.j, h = cur.h;
    Slot nxt;
    const bool more = get_slot<kSrc>(P, W, s_idx + gridDim.x, nlist, nxt);
    bool ok = true;  // every bounded wait of this thread succeeded
    KDA_PT(13);
    ok &= bar_wait(bar_s, par, args.err);
    ok &= bar_wait(bar_p1, par, args.err);
    ok &= bar_wait(bar_p2, par, args.err);
    if (len < kC)  // dO rows past the sequence end hold other tokens: clear them
      for (int it2 = tid; it2 < (kC - len) * 16; it2 += kCT) {
        const int r = 64 + len + (it2 >> 4), q = it2 & 15;
        *reinterpret_cast<uint4 *>(sm + I_STK + sw_chunk(r, q, 192)) = make_uint4(0, 0, 0, 0);
      }
    cp_wait_all();  // G, beta
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(14);

    // ---- tensor-core products ----
    if (tid == 0) {
      // (dX h^T)[r][c] = sum_v dX[r][v] h[c][v] and (dO h^T)[r][c]   (M=64 r, N=128 c, K=128 v)
      const uint32_t id3 = idesc(64, 128, 0, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k) mma(tmem, desc_k16(sbase + I_STK, k, 192), desc_k16(sbase + I_H, k, kD), id3, k > 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + 128, desc_k16(sbase + I_STK + 64 * 128, k, 192), desc_k16(sbase + I_H, k, kD), id3, k > 0);
      // dKhat[r][c] = sum_v D[r][v] dh'[c][v]   (M=64 r, N=128 c, K=128 v)
      const uint32_t id4 = idesc(64, 128, 1, 0), id5 = idesc(128, 128, 1, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k) mma(tmem + 256, desc_mn(sbase + I_DT, k, 8192), desc_k16(sbase + I_DH, k, kD), id4, k > 0);
      // Z[i'][n'] = sum_v [X; D][i'][v] [dO; dD][n'][v]   (M=128, N=128, K=128 v)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem + 384, desc_mn(sbase + I_XT, k, 16384), desc_k16(sbase + I_STK + 64 * 128, k, 192), id5, k > 0);
      commit(bar);
    }
    // meanwhile on the other warps (warp 0 only issues the products): warps 4..7
    // d(2^G_last)[c] = sum_v dh'[c][v] h[c][v]; warps 1..3, 8..15 dv = beta dX and sum_v dX v
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
    for (int r = rw; warp != 0 && (warp < 4 || warp >= 8) && r < kC; r += 11) {  // one warp per row, 4 columns per lane
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
    ok &= bar_wait(bar, par, args.err);
    fence_after();
    __syncthreads();  // products in TMEM; the operand tiles are dead
    KDA_PT(0);

    // ---- raw k, q rows for the decay tiles; dA^T, dAqk^T out of TMEM as hi/lo tiles; gate cumsum ----
    if (tid == 0) {  // raw k, q rows (TMA) into the dead operand tiles
      fence_async_smem();
      mbar_expect_tx(bar_kq, 32768u);
      tma_tile(sbase + C_KRAW, &maps.k, h, t0, bar_kq);
      tma_tile(sbase + C_QRAW, &maps.q, h, t0, bar_kq);
    }
    {
      // Z: lanes 0..63 (i), cols 64..127 (m) = dA^T[i][m]; lanes 64..127, cols 0..63 = dAqk^T[i][r]
      const int cg = warp >> 2, i = 32 * (quarter & 1) + lane;
      const bool qk = quarter >= 2;
      float x[16];
      tmem_ld16(tq + 384u + (qk ? 0u : 64u) + (uint32_t)(16 * cg), x);
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int col = 16 * cg + 8 * hx + e;
          y[e] = (qk && i > col) ? 0.f : x[8 * hx + e];  // dAqk^T[i][r] is a gradient of Aqk only where i <= r
        }
        uint4 hi, lo;
        split8(y, hi, lo);
        const uint32_t off = sw_chunk(i, 2 * cg + hx, kC);
        *reinterpret_cast<uint4 *>(sm + (qk ? C_DQK : C_DAB) + off) = hi;
        *reinterpret_cast<uint4 *>(sm + (qk ? C_DQK : C_DAB) + LO64 + off) = lo;
      }
    }
    // ---- G, block references, decay tiles Kr, Qr, Kc (hi/lo) ----
    if (kGate) {  // the decay from the raw gate
      kgate_tile<kCT>(G, kGLD, len, P.K, j, ga);
      __syncthreads();
    }
    int wide_c = 0;
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
      float rref[4], cref[4];
#pragma unroll
      for (int R = 0; R < 4; ++R) {  // rows past len hold G_last, so the references need no clamping
        const float gref = col[16 * R], gend = col[16 * R + 15];
        wide_c |= !(gref - gend <= kSpanMax);  // (NaN-safe)
        rref[R] = kFix ? gref : 0.5f * (gref + gend);
        cref[R] = kFix ? gend : rref[R];
        vec[(V_RREF + R) * kD + c] = rref[R];
        vec[(V_EREF + R) * kD + c] = exp2f(rref[R]);
        vec[(V_LAM + R) * kD + c] = exp2f(gl - cref[R]);
        if (kFix) vec[(V_CREF + R) * kD + c] = cref[R];
      }
      int p = 0;
#pragma unroll
      for (int R = 1; R < 4; ++R)
#pragma unroll
        for (int I = 0; I < R; ++I) vec[(V_D + p++) * kD + c] = exp2f(rref[R] - cref[I]);
    }
    ok &= bar_wait(bar_kq, par, args.err);  // raw k, q
    if (len < kC) {  // rows past the sequence end hold other tokens: clear them
      zero_tail<kCT>(sm + C_KRAW, len);
      zero_tail<kCT>(sm + C_QRAW, len);
    }
    // a block's decay span is wider than the middle references carry: list the
    // slot for the fix-up launch (whose exact results replace this launch's)
    constexpr bool wide = kFix;
    if (!kFix && __syncthreads_or(wide_c) != 0 && tid == 0) W.wide_grad[atomicAdd(W.flags + 4, 1)] = (int)cur.slot;
    if (kFix) __syncthreads();
    KDA_PT(1);
    {
      const int jj = tid & 15, c0 = jj * 8, rg = tid >> 4, R = rg >> 3;  // two rows per thread
      float rref[8];
#pragma unroll
      for (int e = 0; e < 8; e += 4)
        *reinterpret_cast<float4 *>(rref + e) = *reinterpret_cast<const float4 *>(vec + (V_RREF + R) * kD + c0 + e);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = rg * 2 + rr;
        const uint32_t off = sw_chunk(r, jj, kC);
        float kv[8], qv[8], o[8], e1[8], e2[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + C_KRAW + off), kv);  // raw k, q (zero past len)
        unpack8(*reinterpret_cast<const uint4 *>(sm + C_QRAW + off), qv);
        if (P.l2norm) {  // q/k L2-norm prologue: the row's 16 chunks sit on this half-warp
          float sk = 0.f, sq = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            sk = fmaf(kv[e], kv[e], sk);
            sq = fmaf(qv[e], qv[e], sq);
          }
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
          }
          const float rk = 1.0f / sqrtf(sk + kL2NormEps), rq = 1.0f / sqrtf(sq + kL2NormEps);
          if (jj == 0) {  // the row's inverse norms, for the fused backward and the exact path (rb is free until the dbeta partials)
            rb[r] = rk;
            rb[kC + r] = rq;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            kv[e] *= rk;
            qv[e] *= rq;
          }
        }
        const float *cref = vec + ((kFix ? V_CREF : V_RREF) + R) * kD + c0;  // Gc(R) = Gr(R) outside the fix-up
        *reinterpret_cast<float4 *>(e2) = *reinterpret_cast<const float4 *>(cref);
        *reinterpret_cast<float4 *>(e2 + 4) = *reinterpret_cast<const float4 *>(cref + 4);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float g = G[r * kGLD + c0 + e];
          e1[e] = ex2(g - rref[e]);  // within 2^(+-kSpanMax/2); <= 1 in the fix-up
          e2[e] = ex2(e2[e] - g);    // likewise
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
    KDA_PT(4);
    // ---- pairwise chains: warp owns rows 16B..16B+15 (as r and as i), columns ch0 .. ch0+31 ----
    // Block-pair products are formed in a temporary, scaled by the per-channel
    // factor D_RI in fp32, and added to the accumulators.
    // (row block = the warp's TMEM lane quarter, so that the assembly reads its products from TMEM)
    const int Bk = warp & 3, ch0 = 32 * (warp >> 2);
    const int i8 = lane >> 2, l4 = lane & 3;  // fragment row (and row + 8) and column pair of this lane
    float xr[4][4] = {}, yr[4][4] = {}, xyi[4][4] = {};  // xyi = xi + yi (only their sum is used)
    for (int I = 0; I <= (wide ? Bk - 1 : Bk); ++I) {  // row side: R = Bk, I = 0..Bk (the exact path: I < Bk)
      const float *Dv = (I < Bk) ? vec + (V_D + Bk * (Bk - 1) / 2 + I) * kD : nullptr;  // no factor inside a block
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
    for (int R = wide ? Bk + 1 : Bk; R < 4; ++R) {  // column side: I = Bk, R = Bk..3 (the exact path: R > Bk)
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
    if (wide) {  // the exact path: the sums to true values, plus the diagonal block from pairwise exponents
      const int r0 = 16 * Bk;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c = ch0 + 8 * nt + 2 * l4;
        const float2 gm = *reinterpret_cast<const float2 *>(vec + (V_RREF + Bk) * kD + c);
        const float2 ge = *reinterpret_cast<const float2 *>(vec + (V_CREF + Bk) * kD + c);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = r0 + i8 + 8 * hh;
          const float2 gr = *reinterpret_cast<const float2 *>(G + r * kGLD + c);
          // the row sums carry e1, the column sums e2: multiply them in
          float x0 = xr[nt][2 * hh] * ex2(gr.x - gm.x), x1 = xr[nt][2 * hh + 1] * ex2(gr.y - gm.y);
          float y0 = yr[nt][2 * hh] * ex2(gr.x - gm.x), y1 = yr[nt][2 * hh + 1] * ex2(gr.y - gm.y);
          float z0 = xyi[nt][2 * hh] * ex2(ge.x - gr.x), z1 = xyi[nt][2 * hh + 1] * ex2(ge.y - gr.y);
#pragma unroll 1
          for (int ts = r0; ts < r0 + 16 && ts < len; ++ts) {  // the diagonal block: every exponent <= 0
            const float2 gs = *reinterpret_cast<const float2 *>(G + ts * kGLD + c);
            const float2 kk = raw_row(P, args, t0, h, ts, c, rb, false);
            if (ts <= r) {  // row side, i = ts
              const float f0 = ex2(gr.x - gs.x), f1 = ex2(gr.y - gs.y);
              const float aq = hilo(sm + C_DQK, ts, r);  // dAqk[r][ts]
              y0 = fmaf(aq * kk.x, f0, y0);
              y1 = fmaf(aq * kk.y, f1, y1);
              if (ts < r) {
                const float al = hilo(sm + C_DAB, r, ts);  // dL[r][ts]
                x0 = fmaf(al * kk.x, f0, x0);
                x1 = fmaf(al * kk.y, f1, x1);
              }
            }
            if (ts >= r) {  // column side, r' = ts
              const float f0 = ex2(gs.x - gr.x), f1 = ex2(gs.y - gr.y);
              const float2 qq = raw_row(P, args, t0, h, ts, c, rb, true);
              const float aq = hilo(sm + C_DQK, r, ts);  // dAqk[ts][r]
              z0 = fmaf(aq * qq.x, f0, z0);
              z1 = fmaf(aq * qq.y, f1, z1);
              if (ts > r) {
                const float ax = hilo(sm + C_XB, ts, r);  // X[ts][r]
                z0 = fmaf(ax * kk.x, f0, z0);
                z1 = fmaf(ax * kk.y, f1, z1);
              }
            }
          }
          xr[nt][2 * hh] = x0; xr[nt][2 * hh + 1] = x1;
          yr[nt][2 * hh] = y0; yr[nt][2 * hh + 1] = y1;
          xyi[nt][2 * hh] = z0; xyi[nt][2 * hh + 1] = z1;
        }
      }
    }
    __syncthreads();  // every warp is done with the chain tiles: dL .. T become the assembly scratch
    KDA_PT(5);
    if (more) {  // the next slot's dh', v, A and h columns 64..127 into the dead dAqk^T, X, T, A and dL tiles
      if (tid == 0) mbar_expect_tx(bar_p1, kBytesP1);
      if (lane == 0 && warp >= 1 && warp <= kCopiesP1) {
        fence_async_smem();
        copy_p1(warp - 1, sbase, W, maps, nxt, bar_p1);
      }
    }

    // ---- assembly (fragment element (r, c)), in four passes of 8 columns per warp ----
    // Each pass reads this warp's 16 x 8 blocks of dX h^T (= -dBk), dO h^T (= dQg)
    // and dKhat straight out of tensor memory, in the C-fragment order of the
    // chain accumulators.  Raw k and q are not re-read: every term that needs them
    // is a product with a decay factor that the hi/lo tiles Kr = k e1, Qr = q~ e1,
    // Kc = k e2 hold.  dg = reverse cumsum of dG over the chunk runs once, after
    // the last pass, as column-pair scans over 8-row segments with segment totals
    // exchanged in shared memory.
    float *totC = vec + V_D * kD;  // [4 blocks][128] in the rows of the block factors
    float sg_part = 0.f;            // scalar gate: this warp's share of dg for row 8 * seg + lane (lanes 0..7)
    // segment totals of the dg scan, rows of 128 fp32 (k = 0..14): every vector row
    // but 2^G_last and the four holding totC
    auto tot_row = [&](int k) -> float * {
      return vec + (k == 0 ? V_GL : k < 9 ? V_RREF + (k - 1) : k < 11 ? V_D + 4 + (k - 9) : V_LAM + (k - 11)) * kD;
    };
    const float *dglv = red + 64;
    float bpart[2] = {0.f, 0.f};
    float dotq[2] = {0.f, 0.f}, dotk[2] = {0.f, 0.f};  // kL2: y . dy of rows i8, i8 + 8 of block Bk
    // The assembly: block factors, or the fix-up's true values.
    auto assemble = [&](auto wide_tag) {
      constexpr bool kWide = decltype(wide_tag)::value;
      if (kL2) {
        // per-quarter partial dots [4 column quarters][64 rows]: q in the rows of the last two
        // block factors, k in the unused row and the upper half of the dbeta partials
        float *pdq = vec + (V_D + 4) * kD;
        float *pdk = (warp >> 2) < 2 ? vec + V_GL * kD + (warp >> 2) * kC : rb + 2 * kC + ((warp >> 2) - 2) * kC;
  #pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int c = ch0 + 8 * nt + 2 * l4;
          float px[4], po[4], pk[4];
          {
            const uint32_t tb = tmem + ((uint32_t)(32 * Bk) << 16) + (uint32_t)(ch0 + 8 * nt);
            tmem_ld_frag3(tb, tb + 128u, tb + 256u, px, po, pk);
          }
          const float2 gm2 = *reinterpret_cast<const float2 *>(vec + (V_RREF + Bk) * kD + c);
          const float2 eref2 = *reinterpret_cast<const float2 *>(vec + (V_EREF + Bk) * kD + c);
          const float2 lam2 = *reinterpret_cast<const float2 *>(vec + (V_LAM + Bk) * kD + c);
          const float2 ge2 = kWide ? *reinterpret_cast<const float2 *>(vec + (V_CREF + Bk) * kD + c) : gm2;  // Gc(Bk)
  #pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * Bk + i8 + 8 * hh;
            const float br = beta[r];
            const uint32_t to = sw_off(r, c, kC);
            const float2 krh = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KR + to));
            const float2 krl = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KR + LO128 + to));
            const float2 qrh = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_QR + to));
            const float2 qrl = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_QR + LO128 + to));
            const float2 g2 = *reinterpret_cast<const float2 *>(G + r * kGLD + c);
            const float2 kw = kWide && r < len ? raw_row(P, args, t0, h, r, c, rb, false) : make_float2(0.f, 0.f);
            const float2 qw = kWide && r < len ? raw_row(P, args, t0, h, r, c, rb, true) : make_float2(0.f, 0.f);
  #pragma unroll
            for (int u = 0; u < 2; ++u) {
              const Opnd o = opnd<kWide, true>(u ? krh.y + krl.y : krh.x + krl.x, u ? qrh.y + qrl.y : qrh.x + qrl.x, 0.f,
                                               u ? g2.y : g2.x, u ? gm2.y : gm2.x, u ? ge2.y : ge2.x,
                                               u ? eref2.y : eref2.x, u ? lam2.y : lam2.x, u ? kw.y : kw.x,
                                               u ? qw.y : qw.x);
              const float dq2 = po[2 * hh + u] * (o.e1 * o.eref) + o.e1 * yr[nt][2 * hh + u];
              const float dk2 = pk[2 * hh + u] * (o.e2 * o.lam) - br * (o.e1 * o.eref) * px[2 * hh + u] +
                                br * o.e1 * xr[nt][2 * hh + u] + o.e2 * xyi[nt][2 * hh + u];
              dotq[hh] = fmaf(o.Qr * o.einv, dq2, dotq[hh]);  // y_q = Qr / e1 / qscale and dy_q = qscale dq2
              dotk[hh] = fmaf(o.Kr * o.einv, dk2, dotk[hh]);  // y_k = Kr / e1 and dy_k = dk2
            }
          }
        }
  #pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
  #pragma unroll
          for (int o = 1; o < 4; o <<= 1) {
            dotq[hh] += __shfl_xor_sync(0xffffffffu, dotq[hh], o);
            dotk[hh] += __shfl_xor_sync(0xffffffffu, dotk[hh], o);
          }
          if (l4 == 0) {
            const int r = 16 * Bk + i8 + 8 * hh;
            pdq[(warp >> 2) * kC + r] = dotq[hh];
            pdk[r] = dotk[hh];
          }
        }
        __syncthreads();
  #pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * Bk + i8 + 8 * hh;
          dotq[hh] = pdq[r] + pdq[kC + r] + pdq[2 * kC + r] + pdq[3 * kC + r];
          dotk[hh] = vec[V_GL * kD + r] + vec[V_GL * kD + kC + r] + rb[2 * kC + r] + rb[3 * kC + r];
        }
      }
  #pragma unroll
      for (int g = 0; g < 4; ++g) {
        KDA_PT(9);
        {
          const int nt = g;
          const int c = ch0 + 8 * nt + 2 * l4;
          float px[4], po[4], pk[4];  // element (i8 + 8 hh, c + u) at index 2 hh + u
          {
            const uint32_t tb = tmem + ((uint32_t)(32 * Bk) << 16) + (uint32_t)(ch0 + 8 * nt);
            tmem_ld_frag3(tb, tb + 128u, tb + 256u, px, po, pk);
          }
          const float2 gm2 = *reinterpret_cast<const float2 *>(vec + (V_RREF + Bk) * kD + c);
          const float2 eref2 = *reinterpret_cast<const float2 *>(vec + (V_EREF + Bk) * kD + c);
          const float2 lam2 = *reinterpret_cast<const float2 *>(vec + (V_LAM + Bk) * kD + c);
          const float2 ge2 = kWide ? *reinterpret_cast<const float2 *>(vec + (V_CREF + Bk) * kD + c) : gm2;  // Gc(Bk)
          float cq[2] = {0.f, 0.f};
  #pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r = 16 * Bk + i8 + 8 * hh;
            const float br = beta[r];
            const float2 vq = make_float2(po[2 * hh], po[2 * hh + 1]);
            const float2 vb = make_float2(-px[2 * hh], -px[2 * hh + 1]);
            const float2 vk = make_float2(pk[2 * hh], pk[2 * hh + 1]);
            const uint32_t to = sw_off(r, c, kC);
            uint32_t *krh_p = reinterpret_cast<uint32_t *>(sm + C_KR + to), *krl_p = reinterpret_cast<uint32_t *>(sm + C_KR + LO128 + to);
            uint32_t *qrh_p = reinterpret_cast<uint32_t *>(sm + C_QR + to), *qrl_p = reinterpret_cast<uint32_t *>(sm + C_QR + LO128 + to);
            const float2 krh = unpack_bf16(*krh_p), krl = unpack_bf16(*krl_p);
            const float2 qrh = unpack_bf16(*qrh_p), qrl = unpack_bf16(*qrl_p);
            const float2 kch = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KC + to));
            const float2 kcl = unpack_bf16(*reinterpret_cast<const uint32_t *>(sm + C_KC + LO128 + to));
            const float2 g2 = *reinterpret_cast<const float2 *>(G + r * kGLD + c);
            const float2 kw = kWide && r < len ? raw_row(P, args, t0, h, r, c, rb, false) : make_float2(0.f, 0.f);
            const float2 qw = kWide && r < len ? raw_row(P, args, t0, h, r, c, rb, true) : make_float2(0.f, 0.f);
            float dq2[2], dk2[2], qv[2], pv[2], yq[2], yk[2];  // yq, yk: kL2's normalised rows (yq times qscale)
  #pragma unroll
            for (int u = 0; u < 2; ++u) {
              // k e1, q~ e1, k e2 and the factors (the exact path: k, q~ and true factors)
              const Opnd o = opnd<kWide, kL2>(u ? krh.y + krl.y : krh.x + krl.x, u ? qrh.y + qrl.y : qrh.x + qrl.x,
                                              u ? kch.y + kcl.y : kch.x + kcl.x, u ? g2.y : g2.x, u ? gm2.y : gm2.x,
                                              u ? ge2.y : ge2.x, u ? eref2.y : eref2.x, u ? lam2.y : lam2.x,
                                              u ? kw.y : kw.x, u ? qw.y : qw.x);
              const float Kr = o.Kr, Qr = o.Qr, Kc = o.Kc, e1 = o.e1, e2 = o.e2, eref = o.eref, lam = o.lam;
              const float dQg = u ? vq.y : vq.x, dBk = u ? vb.y : vb.x, dKh = u ? vk.y : vk.x;
              const float gam = e1 * eref, kh = e2 * lam;
              const float xR = xr[nt][2 * hh + u], yR = yr[nt][2 * hh + u];
              const float xyI = xyi[nt][2 * hh + u];
              dq2[u] = dQg * gam + e1 * yR;
              dk2[u] = dKh * kh + br * gam * dBk + br * e1 * xR + e2 * xyI;
              yq[u] = Qr * o.einv;
              yk[u] = Kr * o.einv;
              // dG = Q + P: P (pairwise decay terms and the Khat term) sums to zero over the chunk
              const bool in = r < len;
              qv[u] = in ? kLn2 * (dQg * Qr * eref + br * dBk * Kr * eref) : 0.f;
              pv[u] = in ? kLn2 * (br * Kr * xR + Qr * yR - Kc * xyI - dKh * Kc * lam) : 0.f;
              bpart[hh] += dBk * Kr * eref + Kr * xR;
              cq[u] += dKh * Kc * lam;
            }
            // dG of (r, c) and (r, c + 1) into the Kr (Q part) and Qr (P part) pair slots just read
            *krh_p = __float_as_uint(qv[0]);
            *krl_p = __float_as_uint(qv[1]);
            *qrh_p = __float_as_uint(pv[0]);
            *qrl_p = __float_as_uint(pv[1]);
            if (r < len && c < P.K) {  // (a 64-wide head: the padded channels are not stored)
              const size_t tok = (size_t)(t0 + r);
              if (kL2) {  // dx = r (dy - y (y . dy)), y_q = Qr / e1 / qscale, y_k = Kr / e1
                const float rk = rb[r], rq = rb[kC + r], dq_dot = dotq[hh] / qscale;
                __nv_bfloat16 *pq = (__nv_bfloat16 *)args.dq + (tok * H + h) * P.K + c;
                __nv_bfloat16 *pk = (__nv_bfloat16 *)args.dk + (tok * H + h) * P.K + c;
                *reinterpret_cast<uint32_t *>(pq) = pack_bf16(rq * (dq2[0] * qscale - yq[0] * dq_dot),
                                                            rq * (dq2[1] * qscale - yq[1] * dq_dot));
                *reinterpret_cast<uint32_t *>(pk) = pack_bf16(rk * (dk2[0] - yk[0] * dotk[hh]), rk * (dk2[1] - yk[1] * dotk[hh]));
              } else if (args.partial) {
                float *pq = (float *)args.dq + (tok * HV + j) * P.K + c, *pk = (float *)args.dk + (tok * HV + j) * P.K + c;
                *reinterpret_cast<float2 *>(pq) = make_float2(dq2[0], dq2[1]);  // scaled in the group reduction
                *reinterpret_cast<float2 *>(pk) = make_float2(dk2[0], dk2[1]);
              } else {
                __nv_bfloat16 *pq = (__nv_bfloat16 *)args.dq + (tok * H + h) * P.K + c;
                __nv_bfloat16 *pk = (__nv_bfloat16 *)args.dk + (tok * H + h) * P.K + c;
                *reinterpret_cast<uint32_t *>(pq) = pack_bf16(dq2[0] * qscale, dq2[1] * qscale);
                *reinterpret_cast<uint32_t *>(pk) = pack_bf16(dk2[0], dk2[1]);
              }
            }
          }
  #pragma unroll
          for (int u = 0; u < 2; ++u) {  // column sums of dKhat k khat over the warp's 16 rows
            float cs = cq[u];
            cs += __shfl_xor_sync(0xffffffffu, cs, 4);
            cs += __shfl_xor_sync(0xffffffffu, cs, 8);
            cs += __shfl_xor_sync(0xffffffffu, cs, 16);
            if (i8 == 0) totC[Bk * kD + c + u] = cs;
          }
        }
        KDA_PT(10);
      }
    };
    assemble(BoolC<kFix>{});
    __syncthreads();  // every thread has parked its dG and its Khat column terms
    KDA_PT(11);
    if (more) {  // the Kc tile, G and beta are dead: the next slot's group P2, G and beta
      if (tid == 0) mbar_expect_tx(bar_p2, kBytesP2);
      if (lane == 0 && warp >= 1 && warp <= kCopiesP2) {
        fence_async_smem();
        copy_p2(warp - 1, sbase, W, maps, nxt, bar_p2);
      }
      issue_gate_beta<kScalarGate>(sbase, sm, P, beta, nxt);
    }
    float2 gpb = make_float2(0.f, 0.f);  // kGate: this thread's dbias partials (its column pair)
    float gpa = 0.f;                      //        and dA_log partial
    {  // dg = reverse cumsum of dG: thread = one column pair, one 8-row segment (8 segments)
      const int c = 2 * (tid & 63), seg = tid >> 6, mid = len >> 1;
      // dG of (r, c) and (r, c + 1): Q parts in the Kr hi / lo slots of the pair, P parts in the
      // Qr hi / lo slots (a warp reads one 128-byte row of each: conflict-free)
      float2 q8[8], p8[8];
      float2 tq = make_float2(0.f, 0.f), tp = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t to = sw_off(8 * seg + k, c, kC);
        q8[k] = make_float2(*reinterpret_cast<const float *>(sm + C_KR + to),
                            *reinterpret_cast<const float *>(sm + C_KR + LO128 + to));
        p8[k] = make_float2(*reinterpret_cast<const float *>(sm + C_QR + to),
                            *reinterpret_cast<const float *>(sm + C_QR + LO128 + to));
        tq.x += q8[k].x; tq.y += q8[k].y;
        tp.x += p8[k].x; tp.y += p8[k].y;
      }
      if (seg > 0) *reinterpret_cast<float2 *>(tot_row(seg - 1) + c) = tq;  // Q totals: rows 0..6
      *reinterpret_cast<float2 *>(tot_row(7 + seg) + c) = tp;                // P totals: rows 7..14
      __syncthreads();  // every thread holds its parked dG in registers: the Kr, Qr tiles are dead
      if (more) {  // the next slot's X^T, D^T, dX and the first column halves of dO, dD into them
        if (tid == 0) mbar_expect_tx(bar_s, kBytesS);
        if (lane == 0 && warp >= 1 && warp <= kCopiesS) {
          fence_async_smem();
          copy_s(warp - 1, sbase, W, maps, nxt, bar_s);
        }
      }
      float2 aq = make_float2(0.f, 0.f), aps = aq, app = aq;
#pragma unroll
      for (int s2 = 0; s2 < 8; ++s2) {
        const float2 b = *reinterpret_cast<const float2 *>(tot_row(7 + s2) + c);
        if (s2 > seg) {
          const float2 a = *reinterpret_cast<const float2 *>(tot_row(s2 - 1) + c);
          aq.x += a.x; aq.y += a.y; aps.x += b.x; aps.y += b.y;
        }
        if (s2 < seg) { app.x += b.x; app.y += b.y; }
      }
      float2 ks = make_float2(0.f, 0.f);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float2 t = *reinterpret_cast<const float2 *>(totC + b * kD + c);
        ks.x += t.x; ks.y += t.y;
      }
      // dg_t = sum_{s>=t} dG_s: the Q part and the carried-state decay term
      // from the chunk end; the zero-sum P part from whichever end is nearer
      // (sum_{s>=t} P_s = -sum_{s<t} P_s, the Khat column sum counted at the
      // last row), halving the cancelling terms it sums.
      const float2 gam = *reinterpret_cast<const float2 *>(vec + V_GAML * kD + c);
      const float2 dgl = *reinterpret_cast<const float2 *>(dglv + c);
      const float2 carried = make_float2(kLn2 * gam.x * dgl.x, kLn2 * gam.y * dgl.y);
      float2 pre[8];
      pre[0] = app;
#pragma unroll
      for (int k = 1; k < 8; ++k) pre[k] = make_float2(pre[k - 1].x + p8[k - 1].x, pre[k - 1].y + p8[k - 1].y);
      float2 qs = aq, ps = make_float2(aps.x + kLn2 * ks.x, aps.y + kLn2 * ks.y);
#pragma unroll
      for (int k = 7; k >= 0; --k) {
        const int r = 8 * seg + k;
        qs.x += q8[k].x; qs.y += q8[k].y;
        ps.x += p8[k].x; ps.y += p8[k].y;
        const bool hi = r >= mid;
        const float2 v = make_float2(qs.x + carried.x + (hi ? ps.x : -pre[k].x), qs.y + carried.y + (hi ? ps.y : -pre[k].y));
        if (kScalarGate) {  // dg_t = sum over the channels: this warp's 64 columns, row k's sum kept by lane k
          float t = r < len ? v.x + v.y : 0.f;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
          if (lane == k) sg_part = t;
        } else if (r < len && c < P.K) {  // (a 64-wide head: the padded channels are not stored)
          const size_t e = ((size_t)(t0 + r) * HV + j) * P.K + c;
          if (kGate) {  // da = dG dg/da; the parameter gradients' partials
            const float2 a2 = __ldg(reinterpret_cast<const float2 *>(P.g + e));
            const float sc = kgate_scale(ga, j);
            const float2 d0 = kgate_grad_fast(a2.x + kgate_bias(ga, P.K, j, c), sc, ga.lb);
            const float2 d1 = kgate_grad_fast(a2.y + kgate_bias(ga, P.K, j, c + 1), sc, ga.lb);
            const float2 da = make_float2(v.x * d0.x, v.y * d1.x);
            *reinterpret_cast<float2 *>(args.dg + e) = da;
            gpb.x += da.x;
            gpb.y += da.y;
            gpa = fmaf(v.x, d0.y, fmaf(v.y, d1.y, gpa));
          } else {
            *reinterpret_cast<float2 *>(args.dg + e) = v;
          }
        }
      }
      if (kGate) {
        *reinterpret_cast<float2 *>(sm + C_GPB + (uint32_t)(seg * kD + c) * 4u) = gpb;
        reinterpret_cast<float *>(sm + C_GPA)[tid] = gpa;
      }
    }
    KDA_PT(12);
    KDA_PT(6);
    // dbeta partials: reduce over the 4 lanes sharing a row, then per column half
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float v = bpart[hh];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (l4 == 0) rb[(warp >> 2) * kC + 16 * Bk + i8 + 8 * hh] = v;
    }
    const bool all_ok = __syncthreads_and(ok) != 0;
    KDA_PT(7);
    if (kGate) {  // the slot's partials, summed in a fixed order: dbias per channel, dA_log per slot
      if (tid < kD) {
        const float *gp = reinterpret_cast<const float *>(sm + C_GPB);
        float t = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) t += gp[s * kD + tid];
        W.gpart_b[cur.slot * kD + tid] = t;
      } else if (warp == kD / 32) {
        const float *gp = reinterpret_cast<const float *>(sm + C_GPA);
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < kCT / 32; ++i) t += gp[lane + 32 * i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) W.gpart_a[cur.slot] = t;
      }
    }
    if (tid < kC && tid < len)
      args.dbeta[(size_t)(t0 + tid) * HV + j] = red[tid] + rb[tid] + rb[kC + tid] + rb[2 * kC + tid] + rb[3 * kC + tid];
    if (kScalarGate) {  // the two warps of each 8-row segment add their halves of the 128 channels
      float *part = vec + V_GL * kD;  // [16 warps][8 rows]: the dg scan has read its totals
      if (lane < 8) part[warp * 8 + lane] = sg_part;
      __syncthreads();
      if (tid < kC && tid < len) {
        const int sg = tid >> 3, k = tid & 7;
        args.dg[(size_t)(t0 + tid) * HV + j] = part[(2 * sg) * 8 + k] + part[(2 * sg + 1) * 8 + k];
      }
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

KDA_PT_EXPORT(kda_debug_intra_phase_cycles)

// The per-chunk gradients: the chunk-reference kernel over every slot, this kernel
// over the slots it left (a wide chunk span), then the exact fix-up over the slots
// with a wide 16-token block (none, usually: the CTAs of a list launch read its
// count and leave).
template <bool kSG, bool kL2, bool kGate>
cudaError_t launch_intra(const Problem &P, const GateArgs &ga, const Workspace &W, const IntraArgs &a,
                         const TmaMaps &maps, unsigned grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_intra_tc_kernel<kSG, kL2, kChunkWideList, kGate>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kda_bwd_intra_tc_kernel<kSG, kL2, kFixList, kGate>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  if ((e = launch_intra_chunk(P, ga, W, a, maps, grid, s)) != cudaSuccess) return e;
  KDA_LAUNCH("kda_bwd_intra_tc_block", s,
             kda_bwd_intra_tc_kernel<kSG, kL2, kChunkWideList, kGate><<<grid, kCT, C_SMEM, s>>>(P, W, a, maps, ga));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  KDA_LAUNCH("kda_bwd_intra_tc_fix", s,
             kda_bwd_intra_tc_kernel<kSG, kL2, kFixList, kGate><<<grid, kCT, C_SMEM, s>>>(P, W, a, maps, ga));
  return cudaGetLastError();
}

cudaError_t tc_backward_intra(const Problem &P, const GateArgs &ga, const Workspace &W, const void *dO, void *dv,
                              void *dq, void *dk, float *dg, float *dbeta, int *err, cudaStream_t s) {
  if (P.NC == 0) return cudaSuccess;
  // fp32 partials when several value heads share a q/k head (reduced, and with the L2-norm
  // prologue normalised, per q/k head afterwards); with HV = H the L2-norm backward is fused
  const bool partial = P.HV != P.H, fuse_l2 = P.l2norm && !partial;
  IntraArgs a{(const __nv_bfloat16 *)dO, (__nv_bfloat16 *)dv, partial ? (void *)W.dqp : dq,
              partial ? (void *)W.dkp : dk, dg, dbeta, partial, err};
  TmaMaps maps;
  cudaError_t e = make_tma_maps(P, P.v, dO, &maps);
  if (e != cudaSuccess) return e;
  int nsm = 0;
  if ((e = sm_count(&nsm)) != cudaSuccess) return e;
  const int64_t slots = (int64_t)P.NC * P.HV;
  const unsigned grid = (unsigned)(slots < nsm ? slots : nsm);  // one CTA per SM, persistent over the slots
  if (P.scalar_gate) return fuse_l2 ? launch_intra<true, true, false>(P, ga, W, a, maps, grid, s)
                                    : launch_intra<true, false, false>(P, ga, W, a, maps, grid, s);
  if (ga.on) return fuse_l2 ? launch_intra<false, true, true>(P, ga, W, a, maps, grid, s)
                              : launch_intra<false, false, true>(P, ga, W, a, maps, grid, s);
  return fuse_l2 ? launch_intra<false, true, false>(P, ga, W, a, maps, grid, s)
                 : launch_intra<false, false, false>(P, ga, W, a, maps, grid, s);
}

}  // namespace kda
