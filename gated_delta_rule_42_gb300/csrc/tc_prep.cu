// Per-chunk preparation of the bf16 chunked KDA forward (K, V = 64 or 128, chunk
// 64): everything a chunk step needs that does not depend on v or on the
// carried state, for every (chunk, value head) slot in parallel.
//
// One CTA per slot (three per SM: 75 KB of shared memory):
//  (a) chunk-local cumsum G of the log2 gate and the decay-scaled tiles;
//  (b) the decayed Gram blocks L (strictly lower, beta-scaled) and Aqk (lower),
//      and A = (I + L)^-1 in fp32;
// and writes the slot's tile record: Bk = beta k 2^G, Qg = q~ 2^G,
// Khat = k 2^(G_last - G), Aqk and A (bf16, swizzled operand tiles) and
// 2^G_last (fp32 [K]).  The sequential state kernel and the reverse scan load
// the record with one bulk copy per chunk.
//
// These are the kkt, solve_tril and recompute_w_u steps of the FLA chunk
// pipeline, as listed in the fla-org/flash-linear-attention commit log (PR #1294,
// "[Fix] Use unit KDA gate scale when A_log is omitted"; PR #985, "[Test] Add
// per-kernel torch baselines + tests for GDN kernels"): L = beta-scaled strictly
// lower decayed K K^T, A = (I + L)^-1, w = A Bk and u = A beta v.  Here w and u
// stay factored as A and Bk: the state kernel forms w h and u with tensor-core
// products.
//
// Decay scaling: three kernels, each exact where it runs.
//  - kda_prep_chunk_tc (every slot) splits 2^(G_r - G_i) at the middle m of each
//    channel's range over the chunk: rows carry e1 = 2^(G_r - m) (tiles Kr, Qr),
//    columns e2 = 2^(m - G_i) (tile Kc), and L, Aqk are one tcgen05 product.
//    It needs every channel's chunk span G_first - G_last <= kChunkSpan.
//  - The block-reference kernel (kda_prep_tc_list, over the slots with a wider
//    span) splits at references inside the 16-token blocks: row r of block R
//    carries e1 = 2^(G_r - Gr(R)), column i of block I e2 = 2^(Gc(I) - G_i), and
//    between blocks (R > I) the factor D_RI = 2^(Gr(R) - Gc(I)) <= 1 goes onto the
//    column fragments of 16x16 warp MMAs.  Both references sit in the middle of
//    the block's range, so e1 and e2 stay within 2^(+-kSpanMax/2) while the
//    block's span is at most kSpanMax; a diagonal block needs no factor.
//  - kda_prep_tc_fix (a slot with a wider block: per-token gates averaging below
//    about -12.8, log2) takes each block's first row as Gr and its last as Gc on
//    every channel: e1, e2 <= 1, so the off-diagonal products only underflow
//    where the true product does, and it forms the diagonal blocks exactly from
//    the raw rows, the decay between tokens i and r as the running product of the
//    per-token decays (diag_direct).  Chunk-level tiles there: Bk = beta k e1
//    2^Gr, Qg = q~ e1 2^Gr and Khat = k e2 2^(G_last - Gc); terms below 2^-30 of
//    the largest may flush to zero.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace umma;
using namespace tc;

// Shared-memory map (offsets from the 1024-aligned base).  Kr and Qr are formed
// in place of the raw k and q rows; once every thread has read its G values,
// G's space holds Kc and then L (fp32); once the Gram blocks are done, Kr / Qr's
// hold the inverse scratch.  Every record tile is written straight to global
// memory, so nothing is left to copy out at the end.
constexpr uint32_t P_K = 0;          // k [64][128] bf16 -> Kr -> A (fp32 scratch)
constexpr uint32_t P_Q = 16384;      // q [64][128] bf16 -> Qr -> T (fp32 scratch)
constexpr uint32_t P_G = 32768;      // g -> G fp32 [64][128] (dense rows: a TMA box) -> L fp32 [64][64] | Kc
constexpr uint32_t P_KC = 49152;     // Kc [64][128] bf16 (the upper half of G's space)
constexpr uint32_t P_VEC = 65536;    // fp32 vectors: 18 rows of 128
constexpr uint32_t P_BETA = 74752;   // beta [64]
constexpr uint32_t P_MISC = 75008;   // mbarrier
constexpr uint32_t P_SMEM = P_MISC + 16 + 1024;  // + alignment slack
static_assert(P_SMEM + 1024 <= 233472 / 3, "three CTAs per SM (228 KB, 1 KB reserved per CTA)");
// vector rows: the row references Gr(R) (= Gc(R) in kda_prep_tc), 2^Gr(R) (in
// kda_prep_tc_fix the column references Gc(R) instead), 2^(G_last - Gc(R)), and
// the block-pair factors D_RI = 2^(Gr(R) - Gc(I)) for R > I
constexpr int W_GREF = 0, W_EREF = 4, W_CREF = 4, W_LAM = 8, W_D = 12;
// Widest per-channel decay span (log2) of a 16-token block that the middle
// references carry: e1 and e2 stay within 2^(+-kSpanMax / 2).
constexpr float kSpanMax = 192.f;

// fp32 [64][64] scratch (L, then A): columns XOR-swizzled by 4 * (row % 8), so
// reads of one column across 8 rows and float4 reads of four consecutive
// columns are both free of bank conflicts.
__device__ __forceinline__ int fsw(int r, int c) { return r * kC + (c ^ ((r & 7) << 2)); }

// q/k L2-norm prologue on one row held by the 16 lanes of a half-warp, 8
// channels each: x <- x / sqrt(sum of the row's squares + eps).
__device__ __forceinline__ void l2norm_row16(float (&kv)[8], float (&qv)[8]) {
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
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    kv[e] *= rk;
    qv[e] *= rq;
  }
}

// Phase (a).  Needs k, q, the gate rows and beta of the chunk in shared memory;
// writes G (in place), the vectors, the decay tiles Kr, Qr (in place of k, q)
// and Kc, and the record's Bk, Qg, Khat tiles and 2^G_last straight to global
// memory (rec).  With l2n, the k and q rows are L2-normalised first.  Ends
// with a __syncthreads.  Returns nonzero (every thread, right after the
// cumsum) when a block's span exceeds kSpanMax: the slot is left to the fix-up.
template <bool kGate>
__device__ __forceinline__ int phase_a(unsigned char *sm, int len, const float *beta, unsigned char *rec, bool l2n,
                                       const GateArgs &ga, float qscale, int K, int j) {
  const int tid = threadIdx.x;
  int wide_c = 0;
  float *G = (float *)(sm + P_G);
  float *vec = (float *)(sm + P_VEC);
  if (kGate) {  // the decay from the raw gate (KDA_GATE_IN_KERNEL); value head blockIdx.y
    kgate_tile<kThr>(G, kGT, len, K, j, ga);
    __syncthreads();
  }
  if (tid < kD) {  // one thread per channel (a warp reads 32 consecutive channels: no bank conflicts)
    const int c = tid;
    float col[kC];
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < kC; ++r) col[r] = G[r * kGT + c];
#pragma unroll
    for (int r = 0; r < kC; ++r) {
      if (r < len) s += col[r];
      col[r] = s;
    }
#pragma unroll
    for (int r = 0; r < kC; ++r) G[r * kGT + c] = col[r];
    const float gl = s;
    reinterpret_cast<float *>(rec + kRecGAML)[c] = exp2f(gl);
    float gref[4];
#pragma unroll
    for (int R = 0; R < 4; ++R) {
      // rows past len hold G_last; the middle of the block's range (NaN-safe span test)
      wide_c |= !(col[16 * R] - col[16 * R + 15] <= kSpanMax);
      gref[R] = 0.5f * (col[16 * R] + col[16 * R + 15]);
      vec[(W_GREF + R) * kD + c] = gref[R];
      vec[(W_EREF + R) * kD + c] = exp2f(gref[R]);
      vec[(W_LAM + R) * kD + c] = exp2f(gl - gref[R]);
    }
    // D_RI = 2^(gref_R - gref_I) for the pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
    int p = 0;
#pragma unroll
    for (int R = 1; R < 4; ++R)
#pragma unroll
      for (int I = 0; I < R; ++I) vec[(W_D + p++) * kD + c] = exp2f(gref[R] - gref[I]);
  }
  if (__syncthreads_or(wide_c)) return 1;
  KDA_PT(1);
  // thread: 8 consecutive channels (one 16-byte chunk) of 4 consecutive rows;
  // a half-warp covers one row, so the record stores are whole 128-byte lines
  {
    const int jj = tid & 15, c0 = jj * 8, rg = tid >> 4, R = rg >> 2;
    float gref[8], eref[8], lam[8];
    uint4 kc[4];  // Kc rows, written once every thread has read its G values
#pragma unroll
    for (int e = 0; e < 8; e += 4) {
      *reinterpret_cast<float4 *>(gref + e) = *reinterpret_cast<const float4 *>(vec + (W_GREF + R) * kD + c0 + e);
      *reinterpret_cast<float4 *>(eref + e) = *reinterpret_cast<const float4 *>(vec + (W_EREF + R) * kD + c0 + e);
      *reinterpret_cast<float4 *>(lam + e) = *reinterpret_cast<const float4 *>(vec + (W_LAM + R) * kD + c0 + e);
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = rg * 4 + rr;
      const uint32_t off = sw_chunk(r, jj, kC);
      float kv[8], qv[8], g[8], e1[8], e2[8], o[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + P_K + off), kv);
      unpack8(*reinterpret_cast<const uint4 *>(sm + P_Q + off), qv);
      if (l2n) l2norm_row16(kv, qv);
      *reinterpret_cast<float4 *>(g) = *reinterpret_cast<const float4 *>(G + r * kGT + c0);
      *reinterpret_cast<float4 *>(g + 4) = *reinterpret_cast<const float4 *>(G + r * kGT + c0 + 4);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        e1[e] = ex2(g[e] - gref[e]);  // within 2^(+-kSpanMax/2)
        e2[e] = ex2(gref[e] - g[e]);
      }
      const float br = beta[r];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e1[e];
      *reinterpret_cast<uint4 *>(sm + P_K + off) = pack8(o);  // Kr, in place of k
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e];
      kc[rr] = pack8(o);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = br * kv[e] * e1[e] * eref[e];
      *reinterpret_cast<uint4 *>(rec + kRecBK + off) = pack8(o);  // Bk
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e] * lam[e];
      *reinterpret_cast<uint4 *>(rec + kRecKH + off) = pack8(o);  // Khat
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = qv[e] * qscale * e1[e];
      *reinterpret_cast<uint4 *>(sm + P_Q + off) = pack8(o);  // Qr, in place of q
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] *= eref[e];
      *reinterpret_cast<uint4 *>(rec + kRecQG + off) = pack8(o);  // Qg
    }
    __syncthreads();  // G is dead: its upper half takes Kc
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) *reinterpret_cast<uint4 *>(sm + P_KC + sw_chunk(rg * 4 + rr, jj, kC)) = kc[rr];
  }
  __syncthreads();
  return 0;
}


// ---- 16x16 warp MMAs on fp32 operands split into hi + lo bf16 (the inverse's merges) ----
// Row strides of the fp32 scratch tiles (row-major), chosen so that the fragment loads
// and stores below are free of bank conflicts.
constexpr int kTs16 = 20, kTs8 = 12;
__device__ __forceinline__ void split2(float2 x, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16(x.x, x.y);
  const float2 h = unpack_bf16(hi);
  lo = pack_bf16(x.x - h.x, x.y - h.y);
}
// A fragment (m16n8k16, rows r0 .., columns k0 ..) of an fp32 [64][64] fsw tile, as hi / lo.
__device__ __forceinline__ void frag_a_f32(const float *M, int r0, int k0, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  split2(*reinterpret_cast<const float2 *>(M + fsw(r0 + g, k0 + 2 * q)), hi[0], lo[0]);
  split2(*reinterpret_cast<const float2 *>(M + fsw(r0 + g + 8, k0 + 2 * q)), hi[1], lo[1]);
  split2(*reinterpret_cast<const float2 *>(M + fsw(r0 + g, k0 + 2 * q + 8)), hi[2], lo[2]);
  split2(*reinterpret_cast<const float2 *>(M + fsw(r0 + g + 8, k0 + 2 * q + 8)), hi[3], lo[3]);
}
// B fragment (element (k, n) = M[k0 + k][n0 + n], k < 16, n < 8) of an fp32 fsw tile.
__device__ __forceinline__ void frag_b_fsw(const float *M, int k0, int n0, uint32_t (&hi)[2], uint32_t (&lo)[2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int k = k0 + 2 * q + 8 * h;
    split2(make_float2(M[fsw(k, n0 + g)], M[fsw(k + 1, n0 + g)]), hi[h], lo[h]);
  }
}
// The same from a row-major fp32 scratch tile of row stride ld.
__device__ __forceinline__ void frag_b_rm(const float *M, int ld, int k0, int n0, uint32_t (&hi)[2],
                                          uint32_t (&lo)[2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int k = k0 + 2 * q + 8 * h;
    split2(make_float2(M[k * ld + n0 + g], M[(k + 1) * ld + n0 + g]), hi[h], lo[h]);
  }
}
__device__ __forceinline__ void mma3x(float (&c)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                      const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
  mma16816(c, ah, bh[0], bh[1]);
  mma16816(c, ah, bl[0], bl[1]);
  mma16816(c, al, bh[0], bh[1]);
}
// C fragment (rows r0 + g, r0 + g + 8; columns c0 + 2q, + 1) into a row-major scratch tile ...
__device__ __forceinline__ void store_c(float *M, int ld, int r0, int c0, const float (&c)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  *reinterpret_cast<float2 *>(M + (r0 + g) * ld + c0 + 2 * q) = make_float2(c[0], c[1]);
  *reinterpret_cast<float2 *>(M + (r0 + g + 8) * ld + c0 + 2 * q) = make_float2(c[2], c[3]);
}
// ... or, negated, into an fp32 fsw tile.
__device__ __forceinline__ void store_c_fsw_neg(float *M, int r0, int c0, const float (&c)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  *reinterpret_cast<float2 *>(M + fsw(r0 + g, c0 + 2 * q)) = make_float2(-c[0], -c[1]);
  *reinterpret_cast<float2 *>(M + fsw(r0 + g + 8, c0 + 2 * q)) = make_float2(-c[2], -c[3]);
}

// The inverse A = (I + L)^-1 of L (fp32 in shared memory, strictly lower) and
// its bf16 record tile.  Begins after a __syncthreads that published L.
__device__ __forceinline__ void invert_store(unsigned char *sm, unsigned char *rec) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float *Lf = (float *)(sm + P_G);
  float *Af = (float *)(sm + P_K);  // overwrites Kr (dead)
  float *Tf = (float *)(sm + P_Q);  // overwrites Qr (dead)
  if (warp < 4 && lane < 16) {
    // diagonal block R = warp: lane i computes column i of (I + L_RR)^-1
    const int R = warp, i = lane;
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) a[m] = (m == i) ? 1.f : 0.f;
    // column-oriented substitution: once a[m] is final, subtract its multiples
    // from every later row (independent updates: a short dependency chain);
    // L is read two columns at a time (one float2 per row and column pair)
#pragma unroll
    for (int mg = 0; mg < 8; ++mg) {
      float2 lr[16];
#pragma unroll
      for (int r = 2 * mg + 1; r < 16; ++r)
        lr[r] = *reinterpret_cast<const float2 *>(Lf + fsw(16 * R + r, 16 * R + 2 * mg));
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int m = 2 * mg + mm;
#pragma unroll
        for (int r = m + 1; r < 16; ++r) a[r] = fmaf(-(mm == 0 ? lr[r].x : lr[r].y), a[m], a[r]);
      }
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) Af[fsw(16 * R + m, 16 * R + i)] = a[m];
  }
  for (int e = tid; e < 6 * 256; e += kThr) {  // strictly-upper blocks of A
    const int b = e >> 8, w = e & 255;
    const int R = (b < 3) ? 0 : (b < 5 ? 1 : 2);
    const int I = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
    Af[fsw(16 * R + (w >> 4), 16 * I + (w & 15))] = 0.f;
  }
  __syncthreads();
  KDA_PT(5);
  // Off-diagonal blocks, 32-blocked: A = [[A1, 0], [A21, A2]] with A21 = -A2 L21 A1,
  // where A1 = [[D0, 0], [-D1 L10 D0, D1]] and A2 likewise from D2, D3 (D_R the
  // diagonal-block inverses above).  The products run on 16x16 warp MMAs with each
  // fp32 operand split into a hi and a lo bf16 (hi*hi + hi*lo + lo*hi: about 16
  // mantissa bits, far below the bf16 rounding of the record), each chain inside one
  // warp: A_{R,R-1} = -D_R (L_{R,R-1} D_{R-1}) for R = 1, 3 on warps 0 and 1, then
  // column block w (8 columns) of A21 = -A2 (L21 A1) on warp w < 4.
  if (warp < 2) {
    const int R = 2 * warp + 1;
    float *Ts = Tf + warp * 16 * kTs16;  // L_{R,R-1} D_{R-1}, row-major [16][kTs16]
    uint32_t ah[4], al[4];
    frag_a_f32(Lf, 16 * R, 16 * (R - 1), ah, al);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t bh[2], bl[2];
      frag_b_fsw(Af, 16 * (R - 1), 16 * (R - 1) + 8 * nt, bh, bl);
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma3x(c, ah, al, bh, bl);
      store_c(Ts, kTs16, 0, 8 * nt, c);
    }
    __syncwarp();
    frag_a_f32(Af, 16 * R, 16 * R, ah, al);  // D_R
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t bh[2], bl[2];
      frag_b_rm(Ts, kTs16, 0, 8 * nt, bh, bl);
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma3x(c, ah, al, bh, bl);
      store_c_fsw_neg(Af, 16 * R, 16 * (R - 1) + 8 * nt, c);
    }
  }
  __syncthreads();
  KDA_PT(6);
  if (warp < 4) {
    float *Ts = Tf + 2 * 16 * kTs16 + warp * 32 * kTs8;  // column block w of L21 A1, [32][kTs8]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t ah[4], al[4], bh[2], bl[2];
        frag_a_f32(Lf, 32 + 16 * mt, 16 * ks, ah, al);  // L21
        frag_b_fsw(Af, 16 * ks, 8 * warp, bh, bl);    // A1 (its upper block is zero)
        mma3x(c, ah, al, bh, bl);
      }
      store_c(Ts, kTs8, 16 * mt, 0, c);
    }
    __syncwarp();
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t ah[4], al[4], bh[2], bl[2];
        frag_a_f32(Af, 32 + 16 * mt, 32 + 16 * ks, ah, al);  // A2
        frag_b_rm(Ts, kTs8, 16 * ks, 0, bh, bl);
        mma3x(c, ah, al, bh, bl);
      }
      store_c_fsw_neg(Af, 32 + 16 * mt, 8 * warp, c);
    }
  }
  __syncthreads();
  KDA_PT(8);
  for (int e = tid; e < kC * kC / 8; e += kThr) {  // A -> bf16 tile, 16-byte chunks
    const int r = e >> 3, jj = e & 7;
    float x[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) x[t] = Af[fsw(r, jj * 8 + t)];
    *reinterpret_cast<uint4 *>(rec + kRecAM + sw_chunk(r, jj, kC)) = pack8(x);
  }
}

// Phase (b).  Needs the decay tiles of phase (a); writes the record's Aqk and A
// tiles straight to global memory (rec).
__device__ __forceinline__ void phase_b(unsigned char *sm, const float *beta, unsigned char *rec) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(sm);
  const float *vec = (const float *)(sm + P_VEC);
  float *Lf = (float *)(sm + P_G);  // G is dead
  // Gram blocks: the 10 block pairs R >= I over the 8 warps (the A fragments of
  // a pair serve both 8-column halves: shared-memory wavefronts bound this phase).
  for (int p = warp; p < 10; p += 8) {
    const int R = p >= 6 ? 3 : p >= 3 ? 2 : p >= 1 ? 1 : 0, I = p - R * (R + 1) / 2;
    const float *Dv = (I < R) ? vec + (W_D + R * (R - 1) / 2 + I) * kD : nullptr;
    float accL[2][4] = {}, accQ[2][4] = {};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t ak[4], aq[4], b[4];
      {
        const int row = 16 * R + (lane & 7) + ((lane >> 3) & 1) * 8, jj = 2 * s + (lane >> 4);
        ldsm_x4(sbase + P_K + sw_chunk(row, jj, kC), ak[0], ak[1], ak[2], ak[3]);
        ldsm_x4(sbase + P_Q + sw_chunk(row, jj, kC), aq[0], aq[1], aq[2], aq[3]);
      }
      {
        const int mi = lane >> 3;
        const int row = 16 * I + (lane & 7) + (mi >> 1) * 8, jj = 2 * s + (mi & 1);
        ldsm_x4(sbase + P_KC + sw_chunk(row, jj, kC), b[0], b[1], b[2], b[3]);
      }
      if (Dv != nullptr) {
        const int c0 = 16 * s + (lane & 3) * 2;
        const float2 d01 = *reinterpret_cast<const float2 *>(Dv + c0);
        const float2 d89 = *reinterpret_cast<const float2 *>(Dv + c0 + 8);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = unpack_bf16(b[t]);
          b[t] = (t & 1) ? pack_bf16(f.x * d89.x, f.y * d89.y) : pack_bf16(f.x * d01.x, f.y * d01.y);
        }
      }
      mma16816(accL[0], ak, b[0], b[1]);
      mma16816(accL[1], ak, b[2], b[3]);
      mma16816(accQ[0], aq, b[0], b[1]);
      mma16816(accQ[1], aq, b[2], b[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * R + (lane >> 2) + hh * 8;
        const int i = 16 * I + nt * 8 + (lane & 3) * 2;
        const float br = beta[r];
        const float l0 = (i < r) ? br * accL[nt][2 * hh] : 0.f;
        const float l1 = (i + 1 < r) ? br * accL[nt][2 * hh + 1] : 0.f;
        *reinterpret_cast<float2 *>(Lf + fsw(r, i)) = make_float2(l0, l1);
        const float a0 = (i <= r) ? accQ[nt][2 * hh] : 0.f;
        const float a1 = (i + 1 <= r) ? accQ[nt][2 * hh + 1] : 0.f;
        *reinterpret_cast<uint32_t *>(rec + kRecAQK + sw_off(r, i, kC)) = pack_bf16(a0, a1);
      }
    }
  }
  if (tid < 6 * 32) {  // Aqk blocks above the diagonal (R < I) are zero
    const int b = tid >> 5, w = tid & 31;
    const int R = (b < 3) ? 0 : (b < 5 ? 1 : 2), I = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
    *reinterpret_cast<uint4 *>(rec + kRecAQK + sw_chunk(16 * R + (w >> 1), 2 * I + (w & 1), kC)) = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  KDA_PT(4);
  invert_store(sm, rec);
}

// A slot's k, q and gate rows (TMA; rows past the tensor end arrive as zeros) and
// beta; rows past len cleared.  Ends with a __syncthreads.
__device__ __forceinline__ void load_slot(const Problem &P, const TmaMaps &maps, unsigned char *sm, uint64_t *bar,
                                          uint32_t parity, int *err, int t0, int len, int h, int j) {
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, HV = P.HV;
  float *beta = (float *)(sm + P_BETA);
  if (tid == 0) {
    mbar_expect_tx(bar, 32768u + (P.scalar_gate ? 0u : 32768u));
    tma_tile(sbase + P_K, &maps.k, h, t0, bar);
    tma_tile(sbase + P_Q, &maps.q, h, t0, bar);
    if (!P.scalar_gate) tma_load3(sbase + P_G, &maps.g, 0, j, t0, bar);
  }
  if (P.scalar_gate) {  // one decay per token: repeated over the 128 channels of the gate tile
    float *Gt = (float *)(sm + P_G);
    constexpr int kIt = kC * 32 / kThr;  // float4 stores per thread; all loads go out first
    float x[kIt];
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int r = (tid + u * kThr) >> 5;
      x[u] = r < len ? P.g[(size_t)(t0 + r) * HV + j] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int it = tid + u * kThr, r = it >> 5, c4 = (it & 31) * 4;
      *reinterpret_cast<float4 *>(Gt + r * kGT + c4) = make_float4(x[u], x[u], x[u], x[u]);
    }
  }
  load_beta(P, beta, t0, len, j);
  cp_commit();
  cp_wait_all();
  bar_wait(bar, parity, err);
  if (len < kC) {  // rows past the sequence end hold the next tokens: clear them
    zero_tail(sm + P_K, len);
    zero_tail(sm + P_Q, len);
  }
  __syncthreads();
}

// ---- one decay reference per chunk: the Gram products on tcgen05 ----

// Shared memory of the chunk-reference kernel: the map above, with [Kr; Qr] as one
// 128-row operand in place of k and q (the two 64-column sub-tiles of 128 rows at
// P_K and P_K + 16 KB), a second mbarrier and the tensor-memory slot.
constexpr uint32_t P_BAR2 = P_MISC + 8, P_TSLOT = P_MISC + 16;
constexpr uint32_t P_SMEM_C = P_MISC + 32 + 1024;
static_assert(P_SMEM_C + 1024 <= 233472 / 3, "three CTAs per SM");
static_assert(P_K + 32768 == P_G, "[Kr; Qr] fills the k and q tiles");
// Widest per-channel decay span (log2) of a chunk that one middle reference carries.
constexpr float kChunkSpan = 192.f;
constexpr uint32_t kTmemCols = 64;  // [L | Aqk] rows (M = 128) x 64 columns, per CTA

// One CTA per (chunk, value head) slot, with the pairwise decay 2^(G_r - G_i) split
// at the middle m of each channel's range over the chunk: e1 = 2^(G_r - m) on
// the rows (Kr, Qr), e2 = 2^(m - G_i) on the columns (Kc), both within
// 2^(+-kChunkSpan/2) when every channel's span G_first - G_last is at most
// kChunkSpan.  Then L and Aqk are one tcgen05 product [Kr; Qr] Kc^T (M = 128,
// N = 64, K = 128, fp32 in tensor memory) with no per-block factor.  A slot
// whose span is wider is listed (W.wide_crec, status word 6) for the
// block-reference kernel below.
template <bool kGate>
__global__ void __launch_bounds__(kThr, 3)
kda_prep_chunk_tc_kernel(Problem P, Workspace W, int *err, const __grid_constant__ TmaMaps maps, GateArgs ga) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  const int c_idx = blockIdx.x, j = blockIdx.y;
  const int4 ch = W.chunk[c_idx];
  if (ch.x < 0) return;  // unused chunk slot
  const int t0 = ch.y, len = ch.z;
  const int HV = P.HV, h = j / (HV / P.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t slot = (size_t)c_idx * HV + j;
  float *beta = (float *)(sm + P_BETA);
  float *G = (float *)(sm + P_G);
  float *vec = (float *)(sm + P_VEC);
  uint64_t *bar = (uint64_t *)(sm + P_MISC), *bar_mma = (uint64_t *)(sm + P_BAR2);
  uint32_t *tslot = (uint32_t *)(sm + P_TSLOT);
  KDA_PT_DECL;

  if (tid == 0) {
    bar_init(bar, 1);
    bar_init(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  load_slot(P, maps, sm, bar, 0u, err, t0, len, h, j);
  KDA_PT(0);
  unsigned char *rec = W.tc_tiles + slot * kTileRecord;
  const float qscale = head_qscale(P.K);

  // ---- G, 2^G_last and the reference m = (G_first + G_last) / 2 per channel ----
  if (kGate) {  // the decay from the raw gate (KDA_GATE_IN_KERNEL)
    kgate_tile<kThr>(G, kGT, len, P.K, j, ga);
    __syncthreads();
  }
  int wide_c = 0;
  if (tid < kD) {
    const int c = tid;
    float col[kC];
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < kC; ++r) col[r] = G[r * kGT + c];
#pragma unroll
    for (int r = 0; r < kC; ++r) {
      if (r < len) s += col[r];
      col[r] = s;
    }
#pragma unroll
    for (int r = 0; r < kC; ++r) G[r * kGT + c] = col[r];
    const float gl = s, m = 0.5f * (col[0] + gl);  // rows past len hold G_last
    wide_c = !(col[0] - gl <= kChunkSpan);        // (NaN-safe)
    reinterpret_cast<float *>(rec + kRecGAML)[c] = exp2f(gl);
    vec[W_GREF * kD + c] = m;
    vec[W_EREF * kD + c] = exp2f(m);
    vec[W_LAM * kD + c] = exp2f(gl - m);
  }
  const bool wide = __syncthreads_or(wide_c) != 0;
  KDA_PT(1);
  if (wide) {  // left to the block-reference kernel
    if (tid == 0) W.wide_crec[atomicAdd(W.flags + 6, 1)] = (int)slot;
  } else {
    // ---- tiles: thread = 8 channels (one 16-byte chunk) of 4 rows, a half-warp per row.
    // [Kr; Qr] takes k's and q's place row by row: Kr row r's two sub-tile chunks land on
    // k's row r (channels 0..63) and q's row r (channels 0..63), Qr's on k's and q's row r
    // (channels 64..127) -- all held by the half-warp that reads row r, so a warp barrier
    // between its reads and its writes suffices. ----
    {
      const int jj = tid & 15, c0 = jj * 8, rg = tid >> 4;
      float mv[8], em[8], lm[8];
#pragma unroll
      for (int e = 0; e < 8; e += 4) {
        *reinterpret_cast<float4 *>(mv + e) = *reinterpret_cast<const float4 *>(vec + W_GREF * kD + c0 + e);
        *reinterpret_cast<float4 *>(em + e) = *reinterpret_cast<const float4 *>(vec + W_EREF * kD + c0 + e);
        *reinterpret_cast<float4 *>(lm + e) = *reinterpret_cast<const float4 *>(vec + W_LAM * kD + c0 + e);
      }
      uint4 kc[4];  // Kc rows, written once every thread has read its G values
#pragma unroll 1    // (rolled: the kernel's code stays small; unrolled it stalled on instruction fetch)
      for (int rr = 0; rr < 4; ++rr) {
        const int r = rg * 4 + rr;
        const uint32_t off = sw_chunk(r, jj, kC);
        float kv[8], qv[8], g[8], e1[8], e2[8], o[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + P_K + off), kv);
        unpack8(*reinterpret_cast<const uint4 *>(sm + P_Q + off), qv);
        __syncwarp();  // the half-warp has read row r of k and q
        if (P.l2norm) l2norm_row16(kv, qv);
        *reinterpret_cast<float4 *>(g) = *reinterpret_cast<const float4 *>(G + r * kGT + c0);
        *reinterpret_cast<float4 *>(g + 4) = *reinterpret_cast<const float4 *>(G + r * kGT + c0 + 4);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          e1[e] = ex2(g[e] - mv[e]);  // within 2^(+-kChunkSpan/2)
          e2[e] = ex2(mv[e] - g[e]);
        }
        const float br = beta[r];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = kv[e] * e1[e];
        *reinterpret_cast<uint4 *>(sm + P_K + sw_chunk(r, jj, 2 * kC)) = pack8(o);  // Kr: rows 0..63
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= br * em[e];
        *reinterpret_cast<uint4 *>(rec + kRecBK + off) = pack8(o);  // Bk = beta k 2^G
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e];
        kc[rr] = pack8(o);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= lm[e];
        *reinterpret_cast<uint4 *>(rec + kRecKH + off) = pack8(o);  // Khat = k 2^(G_last - G)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = qv[e] * qscale * e1[e];
        *reinterpret_cast<uint4 *>(sm + P_K + sw_chunk(kC + r, jj, 2 * kC)) = pack8(o);  // Qr: rows 64..127
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= em[e];
        *reinterpret_cast<uint4 *>(rec + kRecQG + off) = pack8(o);  // Qg = q~ 2^G
      }
      __syncthreads();  // G is dead: its upper half takes Kc
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) *reinterpret_cast<uint4 *>(sm + P_KC + sw_chunk(rg * 4 + rr, jj, kC)) = kc[rr];
    }
    fence_async_smem();  // [Kr; Qr] and Kc are read by the tensor core next
    fence_before();
    __syncthreads();
    fence_after();
    KDA_PT(2);
    // ---- [L~ | Aqk][m][i] = sum_c [Kr; Qr][m][c] Kc[i][c]   (M = 128, N = 64, K = 128) ----
    if (tid == 0) {
      const uint32_t id = idesc(128, 64, 0, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma(tmem, desc_k16(sbase + P_K, k, 2 * kC), desc_k16(sbase + P_KC, k, kC), id, k > 0);
      commit(bar_mma);
    }
    bar_wait(bar_mma, 0u, err);
    fence_after();
    {  // warp: lane quarter w % 4 (rows 32 (w % 4) ..), columns 32 (w / 4) ..; L to fp32 shared
       // memory for the inverse (beta-scaled, strictly lower), Aqk (lower) to the record
      const int q4 = warp & 3, c32 = 32 * (warp >> 2), m = 32 * q4 + lane;
      float x[32];
      tmem_ld32(tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)c32, x);
      float *Lf = (float *)(sm + P_G);  // G is dead
      if (m < kC) {
        const int r = m;
        const float br = beta[r];
#pragma unroll
        for (int i4 = 0; i4 < 32; i4 += 4) {
          const int i = c32 + i4;
          *reinterpret_cast<float4 *>(Lf + fsw(r, i)) =
              make_float4(i < r ? br * x[i4] : 0.f, i + 1 < r ? br * x[i4 + 1] : 0.f, i + 2 < r ? br * x[i4 + 2] : 0.f,
                          i + 3 < r ? br * x[i4 + 3] : 0.f);
        }
      } else {
        const int r = m - kC;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = (c32 + 8 * t + e <= r) ? x[8 * t + e] : 0.f;
          *reinterpret_cast<uint4 *>(rec + kRecAQK + sw_chunk(r, (c32 >> 3) + t, kC)) = pack8(y);
        }
      }
    }
    fence_before();
    __syncthreads();
    KDA_PT(4);
    invert_store(sm, rec);
  }
  KDA_PT(10);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_free(tmem, kTmemCols);
  }
  KDA_PT_FLUSH;
}

// The block-reference record kernel (phases (a) and (b) above) over the slots the
// chunk-reference kernel listed (status word 6), walked by the CTAs; a slot with a
// wide 16-token block goes on to the exact fix-up list (status word 3).
template <bool kGate>
__global__ void __launch_bounds__(kThr, 3)
kda_prep_tc_list_kernel(Problem P, Workspace W, int *err, const __grid_constant__ TmaMaps maps, GateArgs ga) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const int nlist = *(volatile const int *)(W.flags + 6);
  if ((int)blockIdx.x >= nlist) return;
  float *beta = (float *)(sm + P_BETA);
  uint64_t *bar = (uint64_t *)(sm + P_MISC);
  if (threadIdx.x == 0) {
    bar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  uint32_t parity = 0;
  for (int i = blockIdx.x; i < nlist; i += gridDim.x, parity ^= 1u) {
    const int s = W.wide_crec[i];
    const int c_idx = s / P.HV, j = s % P.HV, h = j / (P.HV / P.H);
    const int4 ch = W.chunk[c_idx];
    load_slot(P, maps, sm, bar, parity, err, ch.y, ch.z, h, j);
    unsigned char *rec = W.tc_tiles + (size_t)s * kTileRecord;
    if (phase_a<kGate>(sm, ch.z, beta, rec, P.l2norm, ga, head_qscale(P.K), P.K, j)) {
      if (threadIdx.x == 0) W.wide_rec[atomicAdd(W.flags + 3, 1)] = s;
    } else {
      phase_b(sm, beta, rec);
    }
    __syncthreads();  // the shared tiles are free for the next slot
  }
}

// ---- the exact path for slots with a wide block ----

// Phase (a) of the fix-up: phase_a with the block's first row as the row
// reference Gr and its last row as the column reference Gc on every channel,
// so that e1, e2 and every off-diagonal factor are <= 1.
__device__ __forceinline__ void fix_phase_a(unsigned char *sm, int len, const float *beta, unsigned char *rec,
                                            bool l2n, const GateArgs &ga, int j, int K) {
  const int tid = threadIdx.x;
  float *G = (float *)(sm + P_G);
  float *vec = (float *)(sm + P_VEC);
  if (ga.on) {  // the decay from the raw gate (KDA_GATE_IN_KERNEL)
    kgate_tile<kThr>(G, kGT, len, K, j, ga);
    __syncthreads();
  }
  const float qscale = head_qscale(K);
  if (tid < kD) {
    const int c = tid;
    float col[kC];
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < kC; ++r) col[r] = G[r * kGT + c];
#pragma unroll
    for (int r = 0; r < kC; ++r) {
      if (r < len) s += col[r];
      col[r] = s;
    }
#pragma unroll
    for (int r = 0; r < kC; ++r) G[r * kGT + c] = col[r];
    const float gl = s;
    reinterpret_cast<float *>(rec + kRecGAML)[c] = exp2f(gl);
    float gref[4], gend[4];
#pragma unroll
    for (int R = 0; R < 4; ++R) {  // rows past len hold G_last
      gref[R] = col[16 * R];
      gend[R] = col[16 * R + 15];
      vec[(W_GREF + R) * kD + c] = gref[R];
      vec[(W_CREF + R) * kD + c] = gend[R];
      vec[(W_LAM + R) * kD + c] = exp2f(gl - gend[R]);
    }
    int p = 0;  // D_RI = 2^(Gr(R) - Gc(I)) for the pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
#pragma unroll
    for (int R = 1; R < 4; ++R)
#pragma unroll
      for (int I = 0; I < R; ++I) vec[(W_D + p++) * kD + c] = exp2f(gref[R] - gend[I]);
  }
  __syncthreads();
  {
    const int jj = tid & 15, c0 = jj * 8, rg = tid >> 4, R = rg >> 2;
    float gref[8], eref[8], lam[8];
    uint4 kc[4];
#pragma unroll
    for (int e = 0; e < 8; e += 4) {
      *reinterpret_cast<float4 *>(gref + e) = *reinterpret_cast<const float4 *>(vec + (W_GREF + R) * kD + c0 + e);
      *reinterpret_cast<float4 *>(lam + e) = *reinterpret_cast<const float4 *>(vec + (W_LAM + R) * kD + c0 + e);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) eref[e] = ex2(gref[e]);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = rg * 4 + rr;
      const uint32_t off = sw_chunk(r, jj, kC);
      float kv[8], qv[8], g[8], e1[8], e2[8], o[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + P_K + off), kv);
      unpack8(*reinterpret_cast<const uint4 *>(sm + P_Q + off), qv);
      if (l2n) l2norm_row16(kv, qv);
      *reinterpret_cast<float4 *>(g) = *reinterpret_cast<const float4 *>(G + r * kGT + c0);
      *reinterpret_cast<float4 *>(g + 4) = *reinterpret_cast<const float4 *>(G + r * kGT + c0 + 4);
      *reinterpret_cast<float4 *>(e2) = *reinterpret_cast<const float4 *>(vec + (W_CREF + R) * kD + c0);
      *reinterpret_cast<float4 *>(e2 + 4) = *reinterpret_cast<const float4 *>(vec + (W_CREF + R) * kD + c0 + 4);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        e1[e] = ex2(g[e] - gref[e]);  // <= 1
        e2[e] = ex2(e2[e] - g[e]);    // <= 1
      }
      const float br = beta[r];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e1[e];
      *reinterpret_cast<uint4 *>(sm + P_K + off) = pack8(o);  // Kr
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * e2[e];
      kc[rr] = pack8(o);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = br * kv[e] * (e1[e] * eref[e]);
      *reinterpret_cast<uint4 *>(rec + kRecBK + off) = pack8(o);  // Bk
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = kv[e] * (e2[e] * lam[e]);
      *reinterpret_cast<uint4 *>(rec + kRecKH + off) = pack8(o);  // Khat
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = qv[e] * qscale * e1[e];
      *reinterpret_cast<uint4 *>(sm + P_Q + off) = pack8(o);  // Qr
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] *= eref[e];
      *reinterpret_cast<uint4 *>(rec + kRecQG + off) = pack8(o);  // Qg
    }
    __syncthreads();  // G is dead: its upper half takes Kc
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) *reinterpret_cast<uint4 *>(sm + P_KC + sw_chunk(rg * 4 + rr, jj, kC)) = kc[rr];
  }
  __syncthreads();
}

// One diagonal block (R, R) of a slot whose decay span defeats the block
// factors: L_ri = beta_r sum_c k_rc k_ic 2^(G_rc - G_ic) (i < r) and
// Aqk_ri = sum_c q~_rc k_ic 2^(G_rc - G_ic) (i <= r) from the raw rows (L2-
// normalised with l2n), the decay between tokens i and r formed as the running
// product of the per-token decays 2^g_s, s = i+1 .. r (g made from the raw gate
// with the KDA gate inside the op): exact for any gate, it only underflows
// where the true factor does.  One warp; lane l holds channels
// 4l .. 4l+3.  Writes the block's L (fp32, Lf) and Aqk (bf16, rec), zeros above
// the diagonal and past len.
__device__ __noinline__ void diag_direct(const Problem &P, const GateArgs &ga, int t0, int len, int h, int j, int R,
                                         const float *beta, float *Lf, unsigned char *rec) {
  const int lane = threadIdx.x & 31, c0 = lane * 4;
  const float qscale = head_qscale(P.K);
  const __nv_bfloat16 *kp = (const __nv_bfloat16 *)P.k, *qp = (const __nv_bfloat16 *)P.q;
  const bool live = c0 < P.K;  // channels past K (a zero-padded 64-wide head) stay zero
  auto ld4 = [&](const __nv_bfloat16 *base, int r, float (&x)[4]) {  // row r of the chunk, this lane's channels
    const uint2 u = live ? __ldg(reinterpret_cast<const uint2 *>(base + ((size_t)(t0 + r) * P.H + h) * P.K + c0))
                         : make_uint2(0u, 0u);
    const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  };
  // inverse row norms of the q/k L2-norm prologue: row 16R + r's are kept by lane r
  float nk = 1.f, nq = 1.f;
  if (P.l2norm) {
    for (int r = 0; r < 16; ++r) {
      float sk = 0.f, sq = 0.f;
      if (16 * R + r < len) {
        float a[4], b[4];
        ld4(kp, 16 * R + r, a);
        ld4(qp, 16 * R + r, b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sk = fmaf(a[e], a[e], sk);
          sq = fmaf(b[e], b[e], sq);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      if (lane == r) {
        nk = 1.0f / sqrtf(sk + kL2NormEps);
        nq = 1.0f / sqrtf(sq + kL2NormEps);
      }
    }
  }
  for (int i = 0; i < 16 && 16 * R + i < len; ++i) {
    const int ti = 16 * R + i;
    float ki[4], F[4] = {1.f, 1.f, 1.f, 1.f};
    ld4(kp, ti, ki);
    const float nki = __shfl_sync(0xffffffffu, nk, i);
#pragma unroll
    for (int e = 0; e < 4; ++e) ki[e] *= nki;
    for (int r = i; r < 16 && 16 * R + r < len; ++r) {
      const int tr = 16 * R + r;
      if (r > i) {  // F *= 2^g of token tr
        const size_t row = (size_t)(t0 + tr) * P.HV + j;
        if (P.scalar_gate) {
          const float a = exp2f(__ldg(P.g + row));
#pragma unroll
          for (int e = 0; e < 4; ++e) F[e] *= a;
        } else if (live) {
          float4 g4 = __ldg(reinterpret_cast<const float4 *>(P.g + row * P.K + c0));
          if (ga.on) {  // the KDA gate: g holds the raw pre-activations
            const float sc = kgate_scale(ga, j);
            g4.x = kgate_fast(g4.x + kgate_bias(ga, P.K, j, c0), sc, ga.lb);
            g4.y = kgate_fast(g4.y + kgate_bias(ga, P.K, j, c0 + 1), sc, ga.lb);
            g4.z = kgate_fast(g4.z + kgate_bias(ga, P.K, j, c0 + 2), sc, ga.lb);
            g4.w = kgate_fast(g4.w + kgate_bias(ga, P.K, j, c0 + 3), sc, ga.lb);
          }
          F[0] *= exp2f(g4.x); F[1] *= exp2f(g4.y); F[2] *= exp2f(g4.z); F[3] *= exp2f(g4.w);
        }
      }
      float kr[4], qr[4];
      ld4(kp, tr, kr);
      ld4(qp, tr, qr);
      const float nkr = __shfl_sync(0xffffffffu, nk, r), nqr = __shfl_sync(0xffffffffu, nq, r) * qscale;
      float sL = 0.f, sQ = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float f = ki[e] * F[e];
        sL = fmaf(kr[e] * nkr, f, sL);
        sQ = fmaf(qr[e] * nqr, f, sQ);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sL += __shfl_xor_sync(0xffffffffu, sL, o);
        sQ += __shfl_xor_sync(0xffffffffu, sQ, o);
      }
      if (lane == 0) {
        Lf[fsw(tr, ti)] = r > i ? beta[tr] * sL : 0.f;
        *reinterpret_cast<__nv_bfloat16 *>(rec + kRecAQK + sw_off(tr, ti, kC)) = __float2bfloat16_rn(sQ);
      }
    }
  }
  for (int e = lane; e < 256; e += 32) {  // the rest of the block: above the diagonal, or past len
    const int r = e >> 4, i = e & 15, tr = 16 * R + r, ti = 16 * R + i;
    if (i > r || tr >= len || ti >= len) {
      Lf[fsw(tr, ti)] = 0.f;
      *reinterpret_cast<__nv_bfloat16 *>(rec + kRecAQK + sw_off(tr, ti, kC)) = __float2bfloat16_rn(0.f);
    }
  }
}

// Phase (b) of the fix-up: the off-diagonal Gram blocks on the block factors,
// the diagonal ones by diag_direct (warps 4..7), then the inverse.
__device__ __forceinline__ void fix_phase_b(unsigned char *sm, const float *beta, unsigned char *rec,
                                            const Problem &P, const GateArgs &ga, int t0, int len, int h, int j) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(sm);
  const float *vec = (const float *)(sm + P_VEC);
  float *Lf = (float *)(sm + P_G);
  for (int p = warp; p < 10; p += 8) {
    const int R = p >= 6 ? 3 : p >= 3 ? 2 : p >= 1 ? 1 : 0, I = p - R * (R + 1) / 2;
    if (I == R) continue;
    const float *Dv = vec + (W_D + R * (R - 1) / 2 + I) * kD;
    float accL[2][4] = {}, accQ[2][4] = {};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t ak[4], aq[4], b[4];
      {
        const int row = 16 * R + (lane & 7) + ((lane >> 3) & 1) * 8, jj = 2 * s + (lane >> 4);
        ldsm_x4(sbase + P_K + sw_chunk(row, jj, kC), ak[0], ak[1], ak[2], ak[3]);
        ldsm_x4(sbase + P_Q + sw_chunk(row, jj, kC), aq[0], aq[1], aq[2], aq[3]);
      }
      {
        const int mi = lane >> 3;
        const int row = 16 * I + (lane & 7) + (mi >> 1) * 8, jj = 2 * s + (mi & 1);
        ldsm_x4(sbase + P_KC + sw_chunk(row, jj, kC), b[0], b[1], b[2], b[3]);
      }
      const int c0 = 16 * s + (lane & 3) * 2;
      const float2 d01 = *reinterpret_cast<const float2 *>(Dv + c0);
      const float2 d89 = *reinterpret_cast<const float2 *>(Dv + c0 + 8);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = unpack_bf16(b[t]);
        b[t] = (t & 1) ? pack_bf16(f.x * d89.x, f.y * d89.y) : pack_bf16(f.x * d01.x, f.y * d01.y);
      }
      mma16816(accL[0], ak, b[0], b[1]);
      mma16816(accL[1], ak, b[2], b[3]);
      mma16816(accQ[0], aq, b[0], b[1]);
      mma16816(accQ[1], aq, b[2], b[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * R + (lane >> 2) + hh * 8;
        const int i = 16 * I + nt * 8 + (lane & 3) * 2;
        const float br = beta[r];
        *reinterpret_cast<float2 *>(Lf + fsw(r, i)) = make_float2(br * accL[nt][2 * hh], br * accL[nt][2 * hh + 1]);
        *reinterpret_cast<uint32_t *>(rec + kRecAQK + sw_off(r, i, kC)) = pack_bf16(accQ[nt][2 * hh], accQ[nt][2 * hh + 1]);
      }
    }
  }
  if (tid < 6 * 32) {  // Aqk blocks above the diagonal (R < I) are zero
    const int b = tid >> 5, w = tid & 31;
    const int R = (b < 3) ? 0 : (b < 5 ? 1 : 2), I = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
    *reinterpret_cast<uint4 *>(rec + kRecAQK + sw_chunk(16 * R + (w >> 1), 2 * I + (w & 1), kC)) = make_uint4(0, 0, 0, 0);
  }
  if (warp >= 4) diag_direct(P, ga, t0, len, h, j, warp - 4, beta, Lf, rec);
  __syncthreads();
  invert_store(sm, rec);
}

// kda_prep_tc_fix: the slots kda_prep_tc listed, walked by the CTAs, on the
// exact path (with none listed every CTA reads the count and leaves).
__global__ void __launch_bounds__(kThr, 3)
kda_prep_tc_fix_kernel(Problem P, Workspace W, int *err, const __grid_constant__ TmaMaps maps, GateArgs ga) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const int nfix = *(volatile const int *)(W.flags + 3);
  if ((int)blockIdx.x >= nfix) return;
  float *beta = (float *)(sm + P_BETA);
  uint64_t *bar = (uint64_t *)(sm + P_MISC);
  if (threadIdx.x == 0) {
    bar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  uint32_t parity = 0;
  for (int i = blockIdx.x; i < nfix; i += gridDim.x, parity ^= 1u) {
    const int s = W.wide_rec[i];
    const int c_idx = s / P.HV, j = s % P.HV, h = j / (P.HV / P.H);
    const int4 ch = W.chunk[c_idx];
    load_slot(P, maps, sm, bar, parity, err, ch.y, ch.z, h, j);
    unsigned char *rec = W.tc_tiles + (size_t)s * kTileRecord;
    fix_phase_a(sm, ch.z, beta, rec, P.l2norm, ga, j, P.K);
    fix_phase_b(sm, beta, rec, P, ga, ch.y, ch.z, h, j);
    __syncthreads();  // the shared tiles are free for the next slot
  }
}

}  // namespace

KDA_PT_EXPORT(kda_debug_prep_phase_cycles)

cudaError_t tc_prepare(const Problem &P, const GateArgs &ga, const Workspace &W, const TmaMaps &maps, int *err,
                       cudaStream_t s) {
  if (P.NC == 0) return cudaSuccess;
  // the chunk-reference kernel over every slot, the block-reference kernel over the
  // slots it left, the exact fix-up over those with a wide block
  auto fast = ga.on ? kda_prep_chunk_tc_kernel<true> : kda_prep_chunk_tc_kernel<false>;
  auto list = ga.on ? kda_prep_tc_list_kernel<true> : kda_prep_tc_list_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(fast, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM_C);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(list, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kda_prep_tc_fix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
  int nsm = 0;
  if (e == cudaSuccess) e = sm_count(&nsm);
  if (e != cudaSuccess) return e;
  KDA_LAUNCH("kda_prep_tc", s, fast<<<dim3(P.NC, P.HV), kThr, P_SMEM_C, s>>>(P, W, err, maps, ga));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t slots = (int64_t)P.NC * P.HV;
  const unsigned grid = (unsigned)(slots < nsm ? slots : nsm), grid3 = (unsigned)(slots < 3 * nsm ? slots : 3 * nsm);
  KDA_LAUNCH("kda_prep_tc_block", s, list<<<grid3, kThr, P_SMEM, s>>>(P, W, err, maps, ga));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  KDA_LAUNCH("kda_prep_tc_fix", s, kda_prep_tc_fix_kernel<<<grid, kThr, P_SMEM, s>>>(P, W, err, maps, ga));
  return cudaGetLastError();
}

}  // namespace kda
