// fp32 chunked KDA backward: the straightforward kernels.
//
// Recompute-then-differentiate, in the shape of FLA's KDA/GDN backward
// (bwd_dhu = reverse state-gradient scan, then the intra-chunk gradients of
// chunk_bwd_dqkwg / chunk_bwd_dv_local / prepare_wy_repr_bwd through the true
// (I + L)^-1; "[Fix] Use unit KDA gate scale when A_log is omitted",
// fla-org/flash-linear-attention PR #1294, commit log).  The forward quantities
// (G, Aqk, A, w, u, h, D) are recomputed by the forward kernels first.
//
// Per chunk, with dh' the gradient of the chunk-end state:
//   reverse scan: dD = Aqk^T dO + Khat dh' ;  dh = diag(2^G_last) dh' + Qg^T dO - w^T dD
//   intra:  dQg = dO h^T, dAqk = tril(dO D^T), dKhat = D dh'^T, dw = -dD h^T,
//           dA = dD (beta v)^T + dw (beta k 2^G)^T, d(beta v) = A^T dD,
//           d(beta k 2^G) = A^T dw, dL = -tril_{-1}(A^T dA A^T),
//           and the chain through L, Aqk and every 2^(+-G) factor into dk, dq, dbeta, dG;
//   dg = reverse cumsum of dG inside the chunk (G is in log2 units, so each
//   d/dG of 2^x carries ln 2).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kLDT = kChunk + 1;
constexpr int kBV = 32;
constexpr float kLn2 = 0.69314718055994530942f;

size_t dh_smem(int K) {
  return sizeof(float) * (K * kBV + 2 * kChunk * K + 2 * kChunk * kBV + K);
}
size_t bwd_intra_smem(int K) {
  return sizeof(float) * (4 * K * kLDT + 5 * kChunk * kChunk + 2 * kChunk);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
simple_dh_scan_kernel(Problem P, Workspace W, const Tin *__restrict__ dO,
                      const float *__restrict__ dhT, float *__restrict__ dh0) {
  const int n = blockIdx.x, j = blockIdx.y, v0 = blockIdx.z * kBV;
  const int K = P.K, V = P.V, HV = P.HV, H = P.H, h = j / (HV / H);
  const int bv = min(kBV, V - v0);
  const int tid = threadIdx.x;
  const int4 si = W.seq[n];
  const Tin *k = (const Tin *)P.k, *q = (const Tin *)P.q;
  const size_t KV = (size_t)K * V;
  const float scale = 1.0f / sqrtf((float)K);

  extern __shared__ float sm[];
  float *sdh = sm;                  // [K][kBV]
  float *sKh = sdh + K * kBV;       // [64][K]  k 2^(G_last - G)
  float *sQg = sKh + kChunk * K;    // [64][K]  q~ 2^G
  float *sdO = sQg + kChunk * K;    // [64][kBV]
  float *sdD = sdO + kChunk * kBV;  // [64][kBV]
  float *sGl = sdD + kChunk * kBV;  // [K]

  for (int idx = tid; idx < K * kBV; idx += kThreads) {
    const int cc = idx / kBV, x = idx - cc * kBV;
    float val = 0.f;
    if (dhT != nullptr && x < bv) val = dhT[((size_t)n * HV + j) * KV + (size_t)cc * V + v0 + x];
    sdh[idx] = val;
  }
  __syncthreads();
  for (int ci = si.w - 1; ci >= 0; --ci) {
    const int c = si.z + ci;
    const int4 ch = W.chunk[c];
    const int t0 = ch.y, len = ch.z;
    const int64_t slot = (int64_t)c * HV + j;
    const float *Gs = W.G + slot * kChunk * K, *ws = W.w + slot * kChunk * K;
    const float *Aqk = W.Aqk + slot * kChunk * kChunk;
    float *dhs = W.dh + slot * KV;
    float *dDs = W.ddelta + slot * kChunk * V;
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
      const int cc = idx / kBV, x = idx - cc * kBV;
      if (x < bv) dhs[(size_t)cc * V + v0 + x] = sdh[idx];
    }
    for (int idx = tid; idx < kChunk * K; idx += kThreads) {
      const int r = idx / K, cc = idx - r * K;
      float kh = 0.f, qg = 0.f;
      if (r < len) {
        const int64_t e = ((int64_t)(t0 + r) * H + h) * K + cc;
        const float G = Gs[idx];
        kh = ldf(k, e) * exp2f(Gs[(len - 1) * K + cc] - G);
        qg = ldf(q, e) * scale * exp2f(G);
      }
      sKh[idx] = kh;
      sQg[idx] = qg;
    }
    for (int idx = tid; idx < kChunk * kBV; idx += kThreads) {
      const int r = idx / kBV, x = idx - r * kBV;
      sdO[idx] = (r < len && x < bv) ? ldf(dO, ((int64_t)(t0 + r) * HV + j) * V + v0 + x) : 0.f;
    }
    for (int cc = tid; cc < K; cc += kThreads) sGl[cc] = exp2f(Gs[(len - 1) * K + cc]);
    __syncthreads();
    for (int idx = tid; idx < kChunk * kBV; idx += kThreads) {
      const int r = idx / kBV, x = idx - r * kBV;
      float s = 0.f;
      if (r < len && x < bv) {
        for (int i = r; i < len; ++i) s = fmaf(Aqk[i * kChunk + r], sdO[i * kBV + x], s);
        for (int cc = 0; cc < K; ++cc) s = fmaf(sKh[r * K + cc], sdh[cc * kBV + x], s);
      }
      sdD[idx] = s;
      if (x < bv) dDs[r * V + v0 + x] = s;
    }
    __syncthreads();
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
      const int cc = idx / kBV, x = idx - cc * kBV;
      float s = sGl[cc] * sdh[idx];
      for (int r = 0; r < len; ++r) {
        s = fmaf(sQg[r * K + cc], sdO[r * kBV + x], s);
        s = fmaf(-ws[r * K + cc], sdD[r * kBV + x], s);
      }
      sdh[idx] = s;
    }
    __syncthreads();
  }
  if (dh0 != nullptr) {
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
      const int cc = idx / kBV, x = idx - cc * kBV;
      if (x < bv) dh0[((size_t)n * HV + j) * KV + (size_t)cc * V + v0 + x] = sdh[idx];
    }
  }
}

// Intra-chunk backward for one (chunk, value head).  Accumulates the
// per-value-head dq~ and dk partials and dG (in the dg buffer), writes dv and
// dbeta, then turns dG into dg by a reverse cumsum.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
simple_bwd_intra_kernel(Problem P, Workspace W, const Tin *__restrict__ dO, Tin *__restrict__ dv,
                        float *__restrict__ dg, float *__restrict__ dbeta) {
  const int c = blockIdx.x, j = blockIdx.y;
  const int4 ch = W.chunk[c];
  if (ch.x < 0) return;
  const int t0 = ch.y, len = ch.z;
  const int K = P.K, V = P.V, HV = P.HV, H = P.H, h = j / (HV / H);
  const int tid = threadIdx.x;
  const int64_t slot = (int64_t)c * HV + j;
  const Tin *q = (const Tin *)P.q, *k = (const Tin *)P.k, *v = (const Tin *)P.v;
  const float scale = 1.0f / sqrtf((float)K);
  const size_t KV = (size_t)K * V;
  const float *Gs = W.G + slot * kChunk * K;
  const float *hs = W.h + slot * KV, *dhs = W.dh + slot * KV;
  const float *Ds = W.delta + slot * kChunk * V, *dDs = W.ddelta + slot * kChunk * V;
  float *dws = W.dw + slot * kChunk * K;
  float *dqa = W.dqp, *dka = W.dkp, *dga = dg;

  extern __shared__ float sm[];
  float *sk = sm;                       // [K][kLDT]
  float *sq = sk + K * kLDT;            // [K][kLDT] q~
  float *sG = sq + K * kLDT;            // [K][kLDT]
  float *sKd = sG + K * kLDT;           // [K][kLDT] k 2^G
  float *sA = sKd + K * kLDT;           // [64][64]
  float *sQK = sA + kChunk * kChunk;    // [64][64] Aqk
  float *sdA = sQK + kChunk * kChunk;   // [64][64] dA, later dL
  float *sdQK = sdA + kChunk * kChunk;  // [64][64] dAqk
  float *sT = sdQK + kChunk * kChunk;   // [64][64] A^T dA
  float *sb = sT + kChunk * kChunk;     // [64]
  float *sdb = sb + kChunk;             // [64]

  for (int idx = tid; idx < kChunk * K; idx += kThreads) {
    const int r = idx / K, cc = idx - r * K;
    float kv = 0.f, qv = 0.f;
    if (r < len) {
      const int64_t e = ((int64_t)(t0 + r) * H + h) * K + cc;
      kv = ldf(k, e);
      qv = ldf(q, e) * scale;
    }
    const float G = Gs[idx];
    sk[cc * kLDT + r] = kv;
    sq[cc * kLDT + r] = qv;
    sG[cc * kLDT + r] = G;
    sKd[cc * kLDT + r] = kv * exp2f(G);
  }
  for (int p = tid; p < kChunk * kChunk; p += kThreads) {
    sA[p] = W.A[slot * kChunk * kChunk + p];
    sQK[p] = W.Aqk[slot * kChunk * kChunk + p];
  }
  if (tid < kChunk) {
    sb[tid] = (tid < len) ? P.beta[(int64_t)(t0 + tid) * HV + j] : 0.f;
    sdb[tid] = 0.f;
  }
  __syncthreads();

  // Every reduction below runs in a fixed order (no float atomics), so the
  // results are bitwise reproducible.
  const int warp = tid >> 5, lane = tid & 31;
  float *sc = sdQK;  // [64][K] scratch for P1-P2; aliases sdQK and sT, unused until P3
  // P1: terms through h and dh' (thread per (r, c))
  for (int idx = tid; idx < len * K; idx += kThreads) {
    const int r = idx / K, cc = idx - r * K;
    const int64_t t = t0 + r;
    float dQg = 0.f, dKh = 0.f, dwv = 0.f;
    for (int x = 0; x < V; ++x) {
      const float hx = hs[(size_t)cc * V + x];
      dQg = fmaf(ldf(dO, (t * HV + j) * V + x), hx, dQg);
      dKh = fmaf(Ds[r * V + x], dhs[(size_t)cc * V + x], dKh);
      dwv = fmaf(-dDs[r * V + x], hx, dwv);
    }
    const float G = sG[cc * kLDT + r], Gl = sG[cc * kLDT + len - 1];
    const float gam = exp2f(G), e = exp2f(Gl - G);
    const float qg = sq[cc * kLDT + r] * gam, kh = sk[cc * kLDT + r] * e;
    const int64_t ei = (t * HV + j) * K + cc;
    dqa[ei] = dQg * gam;
    dka[ei] = dKh * e;
    dga[ei] = kLn2 * (dQg * qg - dKh * kh);
    dws[r * K + cc] = dwv;
    sc[r * K + cc] = kLn2 * dKh * kh;
  }
  __syncthreads();
  // P2: the decay of the carried state, d(2^G_last) = rowsum(dh' .* h)
  for (int cc = tid; cc < K; cc += kThreads) {
    float s = 0.f;
    for (int x = 0; x < V; ++x) s = fmaf(dhs[(size_t)cc * V + x], hs[(size_t)cc * V + x], s);
    float acc = 0.f;
    for (int r = 0; r < len; ++r) acc += sc[r * K + cc];
    const float Gl = sG[cc * kLDT + len - 1];
    dga[((int64_t)(t0 + len - 1) * HV + j) * K + cc] += acc + kLn2 * exp2f(Gl) * s;
  }
  __syncthreads();
  // P3: dA and dAqk (thread per (r, i))
  for (int p = tid; p < kChunk * kChunk; p += kThreads) {
    const int r = p >> 6, i = p & 63;
    float a = 0.f, aq = 0.f;
    if (r < len && i < len) {
      for (int x = 0; x < V; ++x) a = fmaf(dDs[r * V + x], ldf(v, ((int64_t)(t0 + i) * HV + j) * V + x), a);
      float b = 0.f;
      for (int cc = 0; cc < K; ++cc) b = fmaf(dws[r * K + cc], sKd[cc * kLDT + i], b);
      a = sb[i] * (a + b);
      if (i <= r)
        for (int x = 0; x < V; ++x) aq = fmaf(ldf(dO, ((int64_t)(t0 + r) * HV + j) * V + x), Ds[i * V + x], aq);
    }
    sdA[p] = a;
    sdQK[p] = aq;
  }
  __syncthreads();
  // P4/P5 (one warp per row r): d(beta v) = A^T dD -> dv, dbeta;
  // d(beta k 2^G) = A^T dw -> dk, dbeta, dG
  for (int r = warp; r < len; r += kThreads / 32) {
    float part = 0.f;
    for (int x = lane; x < V; x += 32) {
      float s = 0.f;
      for (int i = r; i < len; ++i) s = fmaf(sA[i * kChunk + r], dDs[i * V + x], s);
      const int64_t e = ((int64_t)(t0 + r) * HV + j) * V + x;
      stf(dv, e, sb[r] * s);
      part = fmaf(s, ldf(v, e), part);
    }
    for (int cc = lane; cc < K; cc += 32) {
      float s = 0.f;
      for (int i = r; i < len; ++i) s = fmaf(sA[i * kChunk + r], dws[i * K + cc], s);
      const float kd = sKd[cc * kLDT + r];
      const int64_t ei = ((int64_t)(t0 + r) * HV + j) * K + cc;
      dka[ei] += sb[r] * exp2f(sG[cc * kLDT + r]) * s;
      dga[ei] += kLn2 * sb[r] * s * kd;
      part = fmaf(s, kd, part);
    }
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) sdb[r] += part;
  }
  // P6: T = A^T dA
  for (int p = tid; p < kChunk * kChunk; p += kThreads) {
    const int r = p >> 6, i = p & 63;
    float s = 0.f;
    for (int m = r; m < kChunk; ++m) s = fmaf(sA[m * kChunk + r], sdA[m * kChunk + i], s);
    sT[p] = s;
  }
  __syncthreads();
  // dL = -tril_{-1}(T A^T)
  for (int p = tid; p < kChunk * kChunk; p += kThreads) {
    const int r = p >> 6, i = p & 63;
    float s = 0.f;
    if (i < r)
      for (int m = 0; m <= i; ++m) s = fmaf(sT[r * kChunk + m], sA[i * kChunk + m], s);
    sdA[p] = -s;
  }
  __syncthreads();
  // P7 (one warp per row r): dbeta from L = beta * KK
  for (int r = warp; r < len; r += kThreads / 32) {
    float part = 0.f;
    for (int i = lane; i < r; i += 32) {
      float kk = 0.f;
      for (int cc = 0; cc < K; ++cc)
        kk = fmaf(sk[cc * kLDT + r] * sk[cc * kLDT + i],
                  exp2f(sG[cc * kLDT + r] - sG[cc * kLDT + i]), kk);
      part = fmaf(sdA[r * kChunk + i], kk, part);
    }
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) sdb[r] += part;
  }
  // P8: row-side pairwise sums (thread per (r, c))
  for (int idx = tid; idx < len * K; idx += kThreads) {
    const int r = idx / K, cc = idx - r * K;
    const float Gr = sG[cc * kLDT + r];
    float xr = 0.f, yr = 0.f;
    for (int i = 0; i <= r; ++i) {
      const float kd = sk[cc * kLDT + i] * exp2f(Gr - sG[cc * kLDT + i]);
      if (i < r) xr = fmaf(sb[r] * sdA[r * kChunk + i], kd, xr);
      yr = fmaf(sdQK[r * kChunk + i], kd, yr);
    }
    const int64_t ei = ((int64_t)(t0 + r) * HV + j) * K + cc;
    dka[ei] += xr;
    dqa[ei] += yr;
    dga[ei] += kLn2 * (sk[cc * kLDT + r] * xr + sq[cc * kLDT + r] * yr);
  }
  __syncthreads();
  // P9: column-side pairwise sums (thread per (i, c))
  for (int idx = tid; idx < len * K; idx += kThreads) {
    const int i = idx / K, cc = idx - i * K;
    const float Gi = sG[cc * kLDT + i];
    float xi = 0.f, yi = 0.f;
    for (int r = i; r < len; ++r) {
      const float d = exp2f(sG[cc * kLDT + r] - Gi);
      if (r > i) xi = fmaf(sb[r] * sdA[r * kChunk + i], sk[cc * kLDT + r] * d, xi);
      yi = fmaf(sdQK[r * kChunk + i], sq[cc * kLDT + r] * d, yi);
    }
    const int64_t ei = ((int64_t)(t0 + i) * HV + j) * K + cc;
    dka[ei] += xi + yi;
    dga[ei] -= kLn2 * sk[cc * kLDT + i] * (xi + yi);
  }
  __syncthreads();
  if (tid < len) dbeta[(int64_t)(t0 + tid) * HV + j] = sdb[tid];
  // dg = reverse cumsum of dG inside the chunk
  for (int cc = tid; cc < K; cc += kThreads) {
    float s = 0.f;
    for (int r = len - 1; r >= 0; --r) {
      const int64_t ei = ((int64_t)(t0 + r) * HV + j) * K + cc;
      s += dga[ei];
      dga[ei] = s;
    }
  }
}

// dq = (sum over the group's value heads of dq~) / sqrt(K); dk = group sum.
template <typename Tin>
__global__ void group_reduce_kernel(Problem P, const float *__restrict__ dqp,
                                    const float *__restrict__ dkp, Tin *__restrict__ dq,
                                    Tin *__restrict__ dk) {
  const int H = P.H, HV = P.HV, K = P.K, r = HV / H;
  int64_t tend = P.Ttot;
  if (P.cu != nullptr) {
    const int64_t e = P.cu[P.N];
    tend = e < 0 ? 0 : (e > P.Ttot ? P.Ttot : e);
  }
  const float scale = 1.0f / sqrtf((float)K);
  const int64_t total = tend * H * K;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = e / ((int64_t)H * K);
    const int rem = (int)(e - t * H * K);
    const int hh = rem / K, cc = rem - hh * K;
    float s1 = 0.f, s2 = 0.f;
    for (int jj = 0; jj < r; ++jj) {
      const int64_t pi = (t * HV + hh * r + jj) * K + cc;
      s1 += dqp[pi];
      s2 += dkp[pi];
    }
    stf(dq, e, s1 * scale);
    stf(dk, e, s2);
  }
}

// The same, four consecutive channels per thread (K a multiple of 4, 16-byte aligned
// partials): each value head's partials in one 16-byte load, the outputs in one store.
// The sums run in the same order, so the results equal the one-channel kernel's bit for bit.
__device__ __forceinline__ void st4(float *p, int64_t i, float4 x) { *reinterpret_cast<float4 *>(p + i) = x; }
__device__ __forceinline__ void st4(__nv_bfloat16 *p, int64_t i, float4 x) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t *>(&a);
  u.y = *reinterpret_cast<const uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p + i) = u;
}
template <typename Tin>
__global__ void group_reduce4_kernel(Problem P, const float4 *__restrict__ dqp, const float4 *__restrict__ dkp,
                                     Tin *__restrict__ dq, Tin *__restrict__ dk) {
  const int H = P.H, HV = P.HV, K4 = P.K / 4, r = HV / H;
  int64_t tend = P.Ttot;
  if (P.cu != nullptr) {
    const int64_t e = P.cu[P.N];
    tend = e < 0 ? 0 : (e > P.Ttot ? P.Ttot : e);
  }
  const float scale = 1.0f / sqrtf((float)P.K);
  const int64_t total = tend * H * K4;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = e / ((int64_t)H * K4);
    const int rem = (int)(e - t * H * K4);
    const int hh = rem / K4, c4 = rem - hh * K4;
    float4 s1 = make_float4(0.f, 0.f, 0.f, 0.f), s2 = s1;
    for (int jj = 0; jj < r; ++jj) {
      const int64_t pi = (t * HV + hh * r + jj) * K4 + c4;
      const float4 a = dqp[pi], b = dkp[pi];
      s1 = make_float4(s1.x + a.x, s1.y + a.y, s1.z + a.z, s1.w + a.w);
      s2 = make_float4(s2.x + b.x, s2.y + b.y, s2.z + b.z, s2.w + b.w);
    }
    st4(dq, 4 * e, make_float4(s1.x * scale, s1.y * scale, s1.z * scale, s1.w * scale));
    st4(dk, 4 * e, s2);
  }
}

template <typename Tin>
cudaError_t run_backward(const Problem &P, const Workspace &W, const void *dO, const float *dhT,
                         void *dq, void *dk, void *dv, float *dg, float *dbeta, float *dh0,
                         bool state_only, cudaStream_t s) {
  cudaError_t e = simple_prepare(P, W, nullptr, s);
  if (e != cudaSuccess) return e;
  const size_t sd = dh_smem(P.K), sb = bwd_intra_smem(P.K);
  e = cudaFuncSetAttribute(simple_dh_scan_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sd);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(simple_bwd_intra_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sb);
  if (e != cudaSuccess) return e;
  if (P.N > 0) {
    KDA_LAUNCH("simple_dh_scan_kernel", s, simple_dh_scan_kernel<Tin><<<dim3(P.N, P.HV, (P.V + kBV - 1) / kBV), kThreads, sd, s>>>(
        P, W, (const Tin *)dO, dhT, dh0));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (state_only) return cudaSuccess;
  if (P.NC > 0) {
    KDA_LAUNCH("simple_bwd_intra_kernel", s, simple_bwd_intra_kernel<Tin><<<dim3(P.NC, P.HV), kThreads, sb, s>>>(P, W, (const Tin *)dO,
                                                                       (Tin *)dv, dg, dbeta));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return launch_group_reduce(P, W.dqp, W.dkp, dq, dk, s);
}

}  // namespace

cudaError_t launch_group_reduce(const Problem &P, const float *dqp, const float *dkp, void *dq, void *dk,
                                cudaStream_t s) {
  if (P.l2norm) return launch_group_reduce_l2norm(P, dqp, dkp, dq, dk, s);
  if (P.Ttot == 0) return cudaSuccess;
  const uintptr_t align = (uintptr_t)dqp | (uintptr_t)dkp | (uintptr_t)dq | (uintptr_t)dk;
  if (P.K % 4 == 0 && (align & 15) == 0) {  // four channels per thread
    const int64_t total4 = P.Ttot * P.H * (P.K / 4);
    int blocks = (int)((total4 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (P.bf16)
      KDA_LAUNCH("group_reduce4_kernel", s, group_reduce4_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
                                                P, (const float4 *)dqp, (const float4 *)dkp, (__nv_bfloat16 *)dq,
                                                (__nv_bfloat16 *)dk));
    else
      KDA_LAUNCH("group_reduce4_kernel", s, group_reduce4_kernel<float><<<blocks, 256, 0, s>>>(
                                                P, (const float4 *)dqp, (const float4 *)dkp, (float *)dq, (float *)dk));
    return cudaGetLastError();
  }
  const int64_t total = P.Ttot * P.H * P.K;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (P.bf16)
    KDA_LAUNCH("group_reduce_kernel", s, group_reduce_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
                                             P, dqp, dkp, (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk));
  else
    KDA_LAUNCH("group_reduce_kernel", s,
               group_reduce_kernel<float><<<blocks, 256, 0, s>>>(P, dqp, dkp, (float *)dq, (float *)dk));
  return cudaGetLastError();
}

cudaError_t simple_backward(const Problem &P, const Workspace &W, const void *dO,
                            const float *dhT, void *dq, void *dk, void *dv, float *dg,
                            float *dbeta, float *dh0, bool state_only, cudaStream_t s) {
  return P.bf16 ? run_backward<__nv_bfloat16>(P, W, dO, dhT, dq, dk, dv, dg, dbeta, dh0, state_only, s)
                : run_backward<float>(P, W, dO, dhT, dq, dk, dv, dg, dbeta, dh0, state_only, s);
}

}  // namespace kda
