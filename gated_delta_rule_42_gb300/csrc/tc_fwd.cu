// Fused bf16 chunked KDA forward on the sm_103a tensor cores (K = V = 128).
//
// One CTA walks the chunks of one (sequence, value head) in order, keeping the
// fp32 state h[K][V] in registers (thread = key channel c, half the value
// columns).  Per 64-token chunk (rows r, i; G = chunk-local cumsum of the log2
// gate; q~ = q / sqrt(K)):
//  (a) G, then the decay-scaled operand tiles.  Pairwise decays 2^(G_r - G_i)
//      are split at the first row of each 16-token block (ref): the row side
//      2^(G_r - G_ref) <= 1 and the column side 2^(G_ref - G_i) <= 2^(15*|g|max),
//      so nothing overflows for gates >= -8 (log2 units); between blocks the
//      per-channel factor D_RI = 2^(G_ref(R) - G_ref(I)) <= 1 is applied to the
//      column operand in registers.  Bk = beta k 2^G, Qg = q~ 2^G and
//      Khat = k 2^(G_last - G) only underflow where the true value is negligible.
//  (b) the strictly-lower decayed beta*K*K^T block L and the lower decayed
//      q~ K^T block Aqk from 16x16 warp MMAs, then A = (I + L)^-1 (fp32: diagonal
//      16-blocks by forward substitution in registers, off-diagonal blocks by
//      A_RI = -A_RR sum_M L_RM A_MI).
//  (c) the state chain on tcgen05 (operands in shared memory, fp32 accumulators
//      in tensor memory):  X^T = (beta v)^T - h^T Bk^T ;  D^T = X^T A^T  (the
//      deltas u - w h) ;  O^T = h^T Qg^T + D^T Aqk^T ;  h <- diag(2^G_last) h + Khat^T D.
// This is the chunk decomposition of the FLA KDA/GDN pipeline (kkt + solve_tril
// + recompute_w_u + fwd_h + fwd_o, named in the commit log of "[Fix] Use unit
// KDA gate scale when A_log is omitted", fla-org/flash-linear-attention PR
// #1294) fused into one pass, with the [K, V] fp32 state held on chip across
// chunks as in the recurrent_kda kernel of "kda in torchtitan (training)".
//
// The same kernel in "states" mode (no output) writes the chunk-start states
// h_c (bf16) for the backward pass.
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kC = 64;      // chunk
constexpr int kD = 128;     // K = V
constexpr int kThr = 256;   // 8 warps
constexpr int kGLD = 132;   // padded fp32 row stride of the gate tile

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KRAW = 0;         // k  [64][128] bf16 SW128
constexpr uint32_t OFF_QRAW = 16384;     // q  [64][128]
constexpr uint32_t OFF_VRAW = 32768;     // v  [64][128]
constexpr uint32_t OFF_GRAW = 49152;     // g -> G  fp32 [64][132]
constexpr uint32_t OFF_BK = 83968;       // beta k 2^G        [64][128]  (MMA B operand)
constexpr uint32_t OFF_QG = 100352;      // q~ 2^G            [64][128]  (MMA B operand)
constexpr uint32_t OFF_KHT = 116736;     // (k 2^(Gl-G))^T    [128][64]  (MMA A operand)
constexpr uint32_t OFF_AQK = 133120;     // Aqk               [64][64]   (MMA B operand)
constexpr uint32_t OFF_AM = 141312;      // A = (I+L)^-1      [64][64]   (MMA B operand)
constexpr uint32_t OFF_U = 149504;       // union (64 KB): phase (a)/(b) | phase (c)
constexpr uint32_t U_KR = 0, U_QR = 16384, U_KC = 32768, U_LF = 49152;  // (a)/(b)
constexpr uint32_t U_AF = 0, U_T = 16384;                              // (b) inverse: A fp32, T fp32
constexpr uint32_t U_HT = 0, U_XT = 32768;                             // (c): h^T [128][128], X^T/D^T [128][64]
constexpr uint32_t OFF_VEC = 215040;     // fp32 vectors, see V_* below (10 KB)
constexpr uint32_t OFF_BETA = 225280;    // beta, two buffers of 64 fp32
constexpr uint32_t OFF_MISC = 225792;    // mbarrier, tmem slot
constexpr uint32_t SMEM_BYTES = 225792 + 64 + 1024;  // + alignment slack
// vector rows (128 floats each)
constexpr int V_GL = 0, V_GAML = 1, V_GREF = 2, V_EREF = 6, V_D = 10, V_LAM = 16;  // 20 rows

constexpr uint32_t TMEM_COLS = 256;  // [0,64) X'^T / O^T, [64,128) D^T, [128,256) Khat^T D

__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void st_zero16(uint32_t dst) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};\n" ::"r"(dst), "r"(0u) : "memory");
}

struct TcArgs {
  __nv_bfloat16 *o;      // [B*T][HV][V] or null
  float *hT;             // [N][HV][K][V] or null
  __nv_bfloat16 *hs;     // chunk-start states [chunk][HV][K][V] bf16 (states mode)
  int *err;              // device error flag
};

// Issue the loads of one chunk's k, q (and g, beta) into the staging tiles.
__device__ __forceinline__ void load_kqg(const Problem &P, unsigned char *sm, int t0, int len, int j,
                                         int h, float *beta_dst) {
  const int tid = threadIdx.x;
  const __nv_bfloat16 *k = (const __nv_bfloat16 *)P.k, *q = (const __nv_bfloat16 *)P.q;
  const uint32_t base = smem_u32(sm);
  for (int it = tid; it < kC * 16; it += kThr) {  // 16-byte chunks of k and q rows
    const int r = it >> 4, jj = it & 15;
    const uint32_t off = sw_chunk(r, jj, kC);
    if (r < len) {
      const size_t row = ((size_t)(t0 + r) * P.H + h) * kD + jj * 8;
      cp16(base + OFF_KRAW + off, k + row);
      cp16(base + OFF_QRAW + off, q + row);
    } else {
      st_zero16(base + OFF_KRAW + off);
      st_zero16(base + OFF_QRAW + off);
    }
  }
  for (int it = tid; it < kC * 32; it += kThr) {  // 16-byte chunks of g rows
    const int r = it >> 5, jj = it & 31;
    const uint32_t dst = base + OFF_GRAW + (uint32_t)(r * kGLD + jj * 4) * 4u;
    if (r < len) cp16(dst, P.g + ((size_t)(t0 + r) * P.HV + j) * kD + jj * 4);
    else st_zero16(dst);
  }
  if (tid < kC) beta_dst[tid] = tid < len ? P.beta[(size_t)(t0 + tid) * P.HV + j] : 0.f;
}

__device__ __forceinline__ void load_v(const Problem &P, unsigned char *sm, int t0, int len, int j) {
  const int tid = threadIdx.x;
  const __nv_bfloat16 *v = (const __nv_bfloat16 *)P.v;
  const uint32_t base = smem_u32(sm);
  for (int it = tid; it < kC * 16; it += kThr) {
    const int r = it >> 4, jj = it & 15;
    const uint32_t off = sw_chunk(r, jj, kC);
    if (r < len) cp16(base + OFF_VRAW + off, v + ((size_t)(t0 + r) * P.HV + j) * kD + jj * 8);
    else st_zero16(base + OFF_VRAW + off);
  }
}

__device__ __forceinline__ float2 ld_bf2(const unsigned char *tile, int r, int c, int R) {
  return unpack_bf16(*reinterpret_cast<const uint32_t *>(tile + sw_off(r, c, R)));
}
__device__ __forceinline__ void st_bf2(unsigned char *tile, int r, int c, int R, float a, float b) {
  *reinterpret_cast<uint32_t *>(tile + sw_off(r, c, R)) = pack_bf16(a, b);
}

template <bool kOut, bool kStates>
__global__ void __launch_bounds__(kThr, 1) kda_fwd_tc_kernel(Problem P, Workspace W, TcArgs args) {
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(sm);
  float *G = (float *)(sm + OFF_GRAW);
  float *vec = (float *)(sm + OFF_VEC);
  float *betab = (float *)(sm + OFF_BETA);
  uint64_t *bar = (uint64_t *)(sm + OFF_MISC);
  uint32_t *tslot = (uint32_t *)(sm + OFF_MISC + 8);
  unsigned char *U = sm + OFF_U;

  const int n = blockIdx.x, j = blockIdx.y;
  const int HV = P.HV, h = j / (HV / P.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, vhalf = warp >> 2;
  const int cown = quarter * 32 + lane;  // key channel / TMEM lane owned in the state epilogues
  const float qscale = 0.08838834764831845f;  // 1/sqrt(128)
  const int4 si = W.seq[n];

  if (tid == 0) {
    bar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  uint32_t phase = 0;

  // state: h[cown][64*vhalf + x], x < 64
  float hreg[64];
  {
    const size_t base = (((size_t)n * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; ++x) hreg[x] = (P.h0 != nullptr) ? P.h0[base + x] : 0.f;
  }

  if (si.w > 0) {
    const int4 ch0 = W.chunk[si.z];
    load_kqg(P, sm, ch0.y, ch0.z, j, h, betab);
    load_v(P, sm, ch0.y, ch0.z, j);
    cp_commit();
  }

  for (int ci = 0; ci < si.w; ++ci) {
    const int cidx = si.z + ci;
    const int4 ch = W.chunk[cidx];
    const int t0 = ch.y, len = ch.z;
    const float *beta = betab + (ci & 1) * kC;
    cp_wait_all();
    __syncthreads();

    // ---------------- (a) gate cumsum and decay factors ----------------
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

    // derived tiles, one 16x16 block per warp iteration in mma-fragment order
    for (int blk = warp; blk < 32; blk += 8) {
      const int rb = (blk >> 3) * 16, cb = (blk & 7) * 16, R = rb >> 4;
      uint32_t khf[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = rb + (lane >> 2) + (m & 1) * 8;
        const int c = cb + (lane & 3) * 2 + (m >> 1) * 8;
        const float2 kv = ld_bf2(sm + OFF_KRAW, r, c, kC);
        const float2 qv = ld_bf2(sm + OFF_QRAW, r, c, kC);
        const float2 g2 = *reinterpret_cast<const float2 *>(G + r * kGLD + c);
        const float gr0 = vec[(V_GREF + R) * kD + c], gr1 = vec[(V_GREF + R) * kD + c + 1];
        const float e1a = exp2f(g2.x - gr0), e1b = exp2f(g2.y - gr1);  // <= 1
        const float e2a = exp2f(gr0 - g2.x), e2b = exp2f(gr1 - g2.y);  // >= 1
        const float era = vec[(V_EREF + R) * kD + c], erb = vec[(V_EREF + R) * kD + c + 1];
        const float la = vec[(V_LAM + R) * kD + c], lb = vec[(V_LAM + R) * kD + c + 1];
        const float br = beta[r];
        if (kOut) st_bf2(U + U_QR, r, c, kC, qv.x * qscale * e1a, qv.y * qscale * e1b);
        st_bf2(U + U_KR, r, c, kC, kv.x * e1a, kv.y * e1b);
        st_bf2(U + U_KC, r, c, kC, kv.x * e2a, kv.y * e2b);
        st_bf2(sm + OFF_BK, r, c, kC, br * kv.x * e1a * era, br * kv.y * e1b * erb);
        if (kOut) st_bf2(sm + OFF_QG, r, c, kC, qv.x * qscale * e1a * era, qv.y * qscale * e1b * erb);
        khf[m] = pack_bf16(kv.x * e2a * la, kv.y * e2b * lb);
      }
      // Khat^T: transposed 16x16 store (rows c, columns r)
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int crow = cb + rr + (mi >> 1) * 8, rcol = rb + (mi & 1) * 8;
        const uint32_t addr = sbase + OFF_KHT + sw_off(crow, rcol, kD);
        asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
                     "r"(khf[0]), "r"(khf[1]), "r"(khf[2]), "r"(khf[3])
                     : "memory");
      }
    }
    __syncthreads();
    // staging k, q, g are consumed: prefetch the next chunk's (v follows after its last use)
    if (ci + 1 < si.w) {
      const int4 nx = W.chunk[cidx + 1];
      load_kqg(P, sm, nx.y, nx.z, j, h, betab + ((ci + 1) & 1) * kC);
      cp_commit();
    }

    // ---------------- (b) decayed Gram blocks and A = (I + L)^-1 ----------------
    float *Lf = (float *)(U + U_LF);
    for (int pr = warp; pr < 16; pr += 8) {
      const int R = pr >> 2, I = pr & 3;
      float accL[2][4] = {}, accQ[2][4] = {};
      if (I <= R) {
        const float *Dv = (I < R) ? vec + (V_D + R * (R - 1) / 2 + I) * kD : nullptr;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t ak[4], aq[4] = {0, 0, 0, 0}, b[4];
          {
            const int row = 16 * R + (lane & 7) + ((lane >> 3) & 1) * 8, jj = 2 * s + (lane >> 4);
            ldsm_x4(sbase + OFF_U + U_KR + sw_chunk(row, jj, kC), ak[0], ak[1], ak[2], ak[3]);
            if (kOut) ldsm_x4(sbase + OFF_U + U_QR + sw_chunk(row, jj, kC), aq[0], aq[1], aq[2], aq[3]);
          }
          {
            const int mi = lane >> 3;
            const int row = 16 * I + (lane & 7) + (mi >> 1) * 8, jj = 2 * s + (mi & 1);
            ldsm_x4(sbase + OFF_U + U_KC + sw_chunk(row, jj, kC), b[0], b[1], b[2], b[3]);
          }
          if (Dv != nullptr) {
            const int c0 = 16 * s + (lane & 3) * 2;
            const float d0 = Dv[c0], d1 = Dv[c0 + 1], d8 = Dv[c0 + 8], d9 = Dv[c0 + 9];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float2 f = unpack_bf16(b[t]);
              b[t] = (t & 1) ? pack_bf16(f.x * d8, f.y * d9) : pack_bf16(f.x * d0, f.y * d1);
            }
          }
          mma16816(accL[0], ak, b[0], b[1]);
          mma16816(accL[1], ak, b[2], b[3]);
          if (kOut) {
            mma16816(accQ[0], aq, b[0], b[1]);
            mma16816(accQ[1], aq, b[2], b[3]);
          }
        }
      }
      // write L (fp32, beta-scaled, strictly lower) and Aqk (bf16, lower incl. diagonal)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = 16 * R + (lane >> 2) + hh * 8;
          const int i = 16 * I + nt * 8 + (lane & 3) * 2;
          const float br = beta[r];
          const float l0 = (i < r) ? br * accL[nt][2 * hh] : 0.f;
          const float l1 = (i + 1 < r) ? br * accL[nt][2 * hh + 1] : 0.f;
          *reinterpret_cast<float2 *>(Lf + r * kC + i) = make_float2(l0, l1);
          if (kOut) {
            const float a0 = (i <= r) ? accQ[nt][2 * hh] : 0.f;
            const float a1 = (i + 1 <= r) ? accQ[nt][2 * hh + 1] : 0.f;
            st_bf2(sm + OFF_AQK, r, i, kC, a0, a1);
          }
        }
      }
    }
    __syncthreads();
    float *Af = (float *)(U + U_AF);  // overwrites Kr (dead)
    float *Tf = (float *)(U + U_T);   // overwrites Qr (dead)
    if (warp < 4 && lane < 16) {
      // diagonal block R = warp: lane i computes column i of (I + L_RR)^-1
      const int R = warp, i = lane;
      float a[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) a[m] = (m == i) ? 1.f : 0.f;
#pragma unroll
      for (int r = 1; r < 16; ++r) {
        float s = a[r];
#pragma unroll
        for (int m = 0; m < r; ++m) s = fmaf(-Lf[(16 * R + r) * kC + 16 * R + m], a[m], s);
        a[r] = s;
      }
#pragma unroll
      for (int m = 0; m < 16; ++m) Af[(16 * R + m) * kC + 16 * R + i] = a[m];
    }
    // zero the strictly-upper blocks of A
    for (int e = tid; e < 6 * 256; e += kThr) {
      const int b = e >> 8, w = e & 255;
      const int R = (b < 3) ? 0 : (b < 5 ? 1 : 2);
      const int I = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
      Af[(16 * R + (w >> 4)) * kC + 16 * I + (w & 15)] = 0.f;
    }
    __syncthreads();
    // off-diagonal blocks by sub-diagonal level: A_RI = -A_RR sum_{M=I}^{R-1} L_RM A_MI
#pragma unroll
    for (int lvl = 1; lvl < 4; ++lvl) {
      const int nb = 4 - lvl;
      for (int e = tid; e < nb * 256; e += kThr) {
        const int I = e >> 8, R = I + lvl, rr = (e >> 4) & 15, ii = e & 15;
        float s = 0.f;
        for (int M = I; M < R; ++M)
#pragma unroll
          for (int m = 0; m < 16; ++m)
            s = fmaf(Lf[(16 * R + rr) * kC + 16 * M + m], Af[(16 * M + m) * kC + 16 * I + ii], s);
        Tf[(I * 16 + rr) * 16 + ii] = s;
      }
      __syncthreads();
      for (int e = tid; e < nb * 256; e += kThr) {
        const int I = e >> 8, R = I + lvl, rr = (e >> 4) & 15, ii = e & 15;
        float s = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) s = fmaf(Af[(16 * R + rr) * kC + 16 * R + m], Tf[(I * 16 + m) * 16 + ii], s);
        Af[(16 * R + rr) * kC + 16 * I + ii] = -s;
      }
      __syncthreads();
    }
    for (int e = tid; e < kC * kC / 2; e += kThr) {
      const int r = e >> 5, i = (e & 31) * 2;
      st_bf2(sm + OFF_AM, r, i, kC, Af[r * kC + i], Af[r * kC + i + 1]);
    }
    __syncthreads();

    // ---------------- (c) state chain on tcgen05 ----------------
    {
      unsigned char *HT = U + U_HT;
#pragma unroll
      for (int x = 0; x < 64; ++x)
        *reinterpret_cast<__nv_bfloat16 *>(HT + sw_off(64 * vhalf + x, cown, kD)) = __float2bfloat16_rn(hreg[x]);
      if (kStates) {
        __nv_bfloat16 *dst = args.hs + (((size_t)cidx * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
        for (int x = 0; x < 64; x += 8) {
          uint4 u;
          u.x = pack_bf16(hreg[x], hreg[x + 1]);
          u.y = pack_bf16(hreg[x + 2], hreg[x + 3]);
          u.z = pack_bf16(hreg[x + 4], hreg[x + 5]);
          u.w = pack_bf16(hreg[x + 6], hreg[x + 7]);
          *reinterpret_cast<uint4 *>(dst + x) = u;
        }
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t aHT = sbase + OFF_U + U_HT, aXT = sbase + OFF_U + U_XT;
    if (tid == 0) {  // X'^T = h^T Bk^T  (M=128 v, N=64 r, K=128 c)
      const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma(tmem, desc_k16(aHT, s, kD), desc_k16(sbase + OFF_BK, s, kC), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    {  // X^T[v][r] = beta_r v[r][v] - X'^T[v][r]
      const int v = quarter * 32 + lane, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)r0, d);
      unsigned char *XT = U + U_XT;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = r0 + q8 * 8 + 2 * e;
          const float v0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_VRAW + sw_off(r, v, kC)));
          const float v1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + OFF_VRAW + sw_off(r + 1, v, kC)));
          pk[e] = pack_bf16(beta[r] * v0 - d[q8 * 8 + 2 * e], beta[r + 1] * v1 - d[q8 * 8 + 2 * e + 1]);
        }
        *reinterpret_cast<uint4 *>(XT + sw_chunk(v, (r0 >> 3) + q8, kD)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (ci + 1 < si.w) {  // v of this chunk is consumed
      const int4 nx = W.chunk[cidx + 1];
      load_v(P, sm, nx.y, nx.z, j);
      cp_commit();
    }
    if (tid == 0) {  // D^T = X^T A^T  (M=128 v, N=64 r, K=64 i)
      const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 64, desc_k16(aXT, s, kD), desc_k16(sbase + OFF_AM, s, kC), id, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    {  // D^T -> bf16 tile (reuses the X^T tile)
      const int v = quarter * 32 + lane, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + 64u + (uint32_t)r0, d);
      unsigned char *DT = U + U_XT;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint4 u;
        u.x = pack_bf16(d[q8 * 8 + 0], d[q8 * 8 + 1]);
        u.y = pack_bf16(d[q8 * 8 + 2], d[q8 * 8 + 3]);
        u.z = pack_bf16(d[q8 * 8 + 4], d[q8 * 8 + 5]);
        u.w = pack_bf16(d[q8 * 8 + 6], d[q8 * 8 + 7]);
        *reinterpret_cast<uint4 *>(DT + sw_chunk(v, (r0 >> 3) + q8, kD)) = u;
      }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {
      if (kOut) {  // O^T = h^T Qg^T + D^T Aqk^T  (M=128 v, N=64 r)
        const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma(tmem, desc_k16(aHT, s, kD), desc_k16(sbase + OFF_QG, s, kC), id, s > 0);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma(tmem, desc_k16(aXT, s, kD), desc_k16(sbase + OFF_AQK, s, kC), id, 1);
      }
      // Khat^T D  (M=128 c, N=128 v, K=64 r)
      const uint32_t id2 = idesc_bf16(128, 128);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma(tmem + 128, desc_k16(sbase + OFF_KHT, s, kD), desc_k16(aXT, s, kD), id2, s > 0);
      commit(bar);
    }
    bar_wait(bar, phase, args.err);
    phase ^= 1;
    fence_after();
    if (kOut) {
      const int v = quarter * 32 + lane, r0 = 32 * vhalf;
      float d[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)r0, d);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int r = r0 + e;
        if (r < len) args.o[((size_t)(t0 + r) * HV + j) * kD + v] = __float2bfloat16_rn(d[e]);
      }
    }
    {
      const float gl = vec[V_GAML * kD + cown];
      float d[32];
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + 128u + (uint32_t)(64 * vhalf + 32 * hx), d);
#pragma unroll
        for (int e = 0; e < 32; ++e) hreg[32 * hx + e] = fmaf(gl, hreg[32 * hx + e], d[e]);
      }
    }
    fence_before();
    __syncthreads();
    fence_after();
  }

  if (args.hT != nullptr) {
    float *dst = args.hT + (((size_t)n * HV + j) * kD + cown) * kD + 64 * vhalf;
#pragma unroll
    for (int x = 0; x < 64; x += 4)
      *reinterpret_cast<float4 *>(dst + x) = make_float4(hreg[x], hreg[x + 1], hreg[x + 2], hreg[x + 3]);
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_free(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t tc_forward(const Problem &P, const Workspace &W, void *o, float *hT, void *hstates,
                       int *err, cudaStream_t s) {
  cudaError_t e = launch_chunk_map(P, W, s);
  if (e != cudaSuccess || P.N == 0) return e;
  TcArgs a{(__nv_bfloat16 *)o, hT, (__nv_bfloat16 *)hstates, err};
  const dim3 grid(P.N, P.HV);
  if (hstates != nullptr) {
    e = cudaFuncSetAttribute(kda_fwd_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    KDA_LAUNCH("kda_fwd_tc_states", s, kda_fwd_tc_kernel<false, true><<<grid, kThr, SMEM_BYTES, s>>>(P, W, a));
  } else {
    e = cudaFuncSetAttribute(kda_fwd_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    KDA_LAUNCH("kda_fwd_tc", s, kda_fwd_tc_kernel<true, false><<<grid, kThr, SMEM_BYTES, s>>>(P, W, a));
  }
  return cudaGetLastError();
}

}  // namespace kda
