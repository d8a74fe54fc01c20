// fp32 chunked KDA forward: the straightforward kernels.
//
// These kernels follow the chunk decomposition of the FLA KDA/GDN pipeline
// (chunk_scaled_dot_kkt + solve_tril + recompute_w_u, then fwd_h, then fwd_o;
// "[Fix] Use unit KDA gate scale when A_log is omitted",
// fla-org/flash-linear-attention PR #1294, commit log) with plain fp32
// arithmetic: SIMT FMAs, pairwise decays 2^(G_r - G_i) formed directly
// (difference first, so nothing overflows for a non-positive gate), the
// unit-lower inverse by forward substitution.  They serve fp32 inputs (whose
// tolerance rules out bf16/tf32 tensor cores) and any K, V <= 128.
//
// Per chunk (rows r, i; G = inclusive cumsum of g inside the chunk; q~ = q/sqrt(K)):
//   L_ri   = beta_r sum_c k_rc k_ic 2^(G_rc - G_ic)      (i < r)
//   Aqk_ri = sum_c q~_rc k_ic 2^(G_rc - G_ic)            (i <= r)
//   A = (I + L)^-1,  w = A (beta k 2^G),  u = A (beta v)
//   scan:   D = u - w h ;  h <- diag(2^G_last) h + (k 2^(G_last - G))^T D
//   output: o = (q~ 2^G) h + Aqk D
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kLDT = kChunk + 1;  // channel-major shared tiles [K][65]: conflict-free rows
constexpr int kBV = 32;           // value columns per scan block

size_t intra_smem(int K, int V) {
  return sizeof(float) * (3 * K * kLDT + kChunk * V + 3 * kChunk * kChunk + kChunk);
}
size_t scan_smem(int K) {
  return sizeof(float) * (K * kBV + kChunk * K + kChunk * kBV + K);
}
size_t out_smem(int K, int V) {
  return sizeof(float) * (kChunk * K + kChunk * kChunk + kChunk * V);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) simple_intra_kernel(Problem P, Workspace W) {
  const int c = blockIdx.x, j = blockIdx.y;
  const int4 ch = W.chunk[c];
  if (ch.x < 0) return;
  const int t0 = ch.y, len = ch.z;
  const int K = P.K, V = P.V, HV = P.HV, H = P.H, h = j / (HV / H);
  const int tid = threadIdx.x;
  const int64_t slot = (int64_t)c * HV + j;
  const Tin *q = (const Tin *)P.q, *k = (const Tin *)P.k, *v = (const Tin *)P.v;
  const float scale = 1.0f / sqrtf((float)K);

  extern __shared__ float sm[];
  float *sk = sm;                     // [K][kLDT]  k
  float *sq = sk + K * kLDT;          // [K][kLDT]  q~, later beta k 2^G
  float *sG = sq + K * kLDT;          // [K][kLDT]  G
  float *sv = sG + K * kLDT;          // [64][V]
  float *sL = sv + kChunk * V;        // [64][64]
  float *sQK = sL + kChunk * kChunk;  // [64][64]
  float *sA = sQK + kChunk * kChunk;  // [64][64]
  float *sb = sA + kChunk * kChunk;   // [64]

  for (int idx = tid; idx < kChunk * K; idx += kThreads) {
    const int r = idx / K, cc = idx - r * K;
    float kv = 0.f, qv = 0.f, gv = 0.f;
    if (r < len) {
      const int64_t t = t0 + r;
      kv = ldf(k, (t * H + h) * K + cc);
      qv = ldf(q, (t * H + h) * K + cc) * scale;
      gv = P.g[(t * HV + j) * K + cc];
    }
    sk[cc * kLDT + r] = kv;
    sq[cc * kLDT + r] = qv;
    sG[cc * kLDT + r] = gv;
  }
  for (int idx = tid; idx < kChunk * V; idx += kThreads) {
    const int r = idx / V, x = idx - r * V;
    sv[idx] = (r < len) ? ldf(v, ((int64_t)(t0 + r) * HV + j) * V + x) : 0.f;
  }
  if (tid < kChunk) sb[tid] = (tid < len) ? P.beta[(int64_t)(t0 + tid) * HV + j] : 0.f;
  __syncthreads();

  // chunk-local inclusive cumsum; padded rows repeat the chunk's last value
  for (int cc = tid; cc < K; cc += kThreads) {
    float s = 0.f;
    for (int r = 0; r < kChunk; ++r) {
      if (r < len) s += sG[cc * kLDT + r];
      sG[cc * kLDT + r] = s;
    }
  }
  __syncthreads();

  // decayed Gram blocks
  for (int p = tid; p < kChunk * kChunk; p += kThreads) {
    const int r = p >> 6, i = p & 63;
    float kk = 0.f, qk = 0.f;
    if (i <= r && r < len) {
      for (int cc = 0; cc < K; ++cc) {
        const float d = exp2f(sG[cc * kLDT + r] - sG[cc * kLDT + i]);
        const float ki = sk[cc * kLDT + i] * d;
        kk = fmaf(sk[cc * kLDT + r], ki, kk);
        qk = fmaf(sq[cc * kLDT + r], ki, qk);
      }
    }
    sL[p] = (i < r) ? sb[r] * kk : 0.f;
    sQK[p] = (i <= r) ? qk : 0.f;
    sA[p] = (r == i) ? 1.f : 0.f;
  }
  __syncthreads();

  // A = (I + L)^-1 by forward substitution: A_ri = -sum_{i<=m<r} L_rm A_mi
  for (int r = 1; r < kChunk; ++r) {
    if (tid < r) {
      float s = 0.f;
      for (int m = tid; m < r; ++m) s = fmaf(sL[r * kChunk + m], sA[m * kChunk + tid], s);
      sA[r * kChunk + tid] = -s;
    }
    __syncthreads();
  }

  // beta k 2^G (channel-major, reusing the q~ tile)
  for (int idx = tid; idx < kChunk * K; idx += kThreads) {
    const int cc = idx / kChunk, r = idx - cc * kChunk;
    sq[cc * kLDT + r] = sb[r] * sk[cc * kLDT + r] * exp2f(sG[cc * kLDT + r]);
  }
  __syncthreads();

  float *wout = W.w + slot * kChunk * K;
  float *Gout = W.G + slot * kChunk * K;
  for (int idx = tid; idx < kChunk * K; idx += kThreads) {
    const int r = idx / K, cc = idx - r * K;
    float s = 0.f;
    for (int i = 0; i <= r; ++i) s = fmaf(sA[r * kChunk + i], sq[cc * kLDT + i], s);
    wout[idx] = s;
    Gout[idx] = sG[cc * kLDT + r];
  }
  float *uout = W.u + slot * kChunk * V;
  for (int idx = tid; idx < kChunk * V; idx += kThreads) {
    const int r = idx / V, x = idx - r * V;
    float s = 0.f;
    for (int i = 0; i <= r; ++i) s = fmaf(sA[r * kChunk + i], sb[i] * sv[i * V + x], s);
    uout[idx] = s;
  }
  float *Aqk = W.Aqk + slot * kChunk * kChunk, *Ao = W.A + slot * kChunk * kChunk;
  for (int p = tid; p < kChunk * kChunk; p += kThreads) {
    Aqk[p] = sQK[p];
    Ao[p] = sA[p];
  }
}

// Inter-chunk state scan over one (sequence, value head, 32-column block).
// Stores the chunk-start state h_c and the deltas D_c of every chunk.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
simple_scan_kernel(Problem P, Workspace W, float *__restrict__ hT) {
  const int n = blockIdx.x, j = blockIdx.y, v0 = blockIdx.z * kBV;
  const int K = P.K, V = P.V, HV = P.HV, H = P.H, h = j / (HV / H);
  const int bv = min(kBV, V - v0);
  const int tid = threadIdx.x;
  const int4 si = W.seq[n];
  const Tin *k = (const Tin *)P.k;
  const size_t KV = (size_t)K * V;

  extern __shared__ float sm[];
  float *sh = sm;                  // [K][kBV]
  float *sKh = sh + K * kBV;       // [64][K]  k 2^(G_last - G)
  float *sD = sKh + kChunk * K;    // [64][kBV]
  float *sGl = sD + kChunk * kBV;  // [K]      2^G_last

  for (int idx = tid; idx < K * kBV; idx += kThreads) {
    const int cc = idx / kBV, x = idx - cc * kBV;
    float val = 0.f;
    if (P.h0 != nullptr && x < bv) val = P.h0[((size_t)n * HV + j) * KV + (size_t)cc * V + v0 + x];
    sh[idx] = val;
  }
  __syncthreads();
  for (int ci = 0; ci < si.w; ++ci) {
    const int c = si.z + ci;
    const int4 ch = W.chunk[c];
    const int t0 = ch.y, len = ch.z;
    const int64_t slot = (int64_t)c * HV + j;
    float *hs = W.h + slot * KV;
    const float *ws = W.w + slot * kChunk * K, *us = W.u + slot * kChunk * V;
    const float *Gs = W.G + slot * kChunk * K;
    float *Ds = W.delta + slot * kChunk * V;
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
      const int cc = idx / kBV, x = idx - cc * kBV;
      if (x < bv) hs[(size_t)cc * V + v0 + x] = sh[idx];
    }
    for (int idx = tid; idx < kChunk * kBV; idx += kThreads) {
      const int r = idx / kBV, x = idx - r * kBV;
      float d = 0.f;
      if (r < len && x < bv) {
        d = us[r * V + v0 + x];
        for (int cc = 0; cc < K; ++cc) d = fmaf(-ws[r * K + cc], sh[cc * kBV + x], d);
      }
      sD[idx] = d;
      if (x < bv) Ds[r * V + v0 + x] = d;
    }
    for (int idx = tid; idx < kChunk * K; idx += kThreads) {
      const int r = idx / K, cc = idx - r * K;
      float kh = 0.f;
      if (r < len)
        kh = ldf(k, ((int64_t)(t0 + r) * H + h) * K + cc) *
             exp2f(Gs[(len - 1) * K + cc] - Gs[r * K + cc]);
      sKh[idx] = kh;
    }
    for (int cc = tid; cc < K; cc += kThreads) sGl[cc] = exp2f(Gs[(len - 1) * K + cc]);
    __syncthreads();
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
      const int cc = idx / kBV, x = idx - cc * kBV;
      float s = sGl[cc] * sh[idx];
      for (int r = 0; r < len; ++r) s = fmaf(sKh[r * K + cc], sD[r * kBV + x], s);
      sh[idx] = s;
    }
    __syncthreads();
  }
  if (hT != nullptr) {
    for (int idx = tid; idx < K * kBV; idx += kThreads) {
      const int cc = idx / kBV, x = idx - cc * kBV;
      if (x < bv) hT[((size_t)n * HV + j) * KV + (size_t)cc * V + v0 + x] = sh[idx];
    }
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
simple_output_kernel(Problem P, Workspace W, Tin *__restrict__ o) {
  const int c = blockIdx.x, j = blockIdx.y;
  const int4 ch = W.chunk[c];
  if (ch.x < 0) return;
  const int t0 = ch.y, len = ch.z;
  const int K = P.K, V = P.V, HV = P.HV, H = P.H, h = j / (HV / H);
  const int tid = threadIdx.x;
  const int64_t slot = (int64_t)c * HV + j;
  const Tin *q = (const Tin *)P.q;
  const float scale = 1.0f / sqrtf((float)K);
  const float *Gs = W.G + slot * kChunk * K, *hs = W.h + slot * (size_t)K * V;

  extern __shared__ float sm[];
  float *sQg = sm;                       // [64][K]
  float *sQK = sQg + kChunk * K;         // [64][64]
  float *sD = sQK + kChunk * kChunk;     // [64][V]
  for (int idx = tid; idx < kChunk * K; idx += kThreads) {
    const int r = idx / K, cc = idx - r * K;
    sQg[idx] = (r < len) ? ldf(q, ((int64_t)(t0 + r) * H + h) * K + cc) * scale * exp2f(Gs[idx]) : 0.f;
  }
  for (int p = tid; p < kChunk * kChunk; p += kThreads) sQK[p] = W.Aqk[slot * kChunk * kChunk + p];
  for (int idx = tid; idx < kChunk * V; idx += kThreads) sD[idx] = W.delta[slot * kChunk * V + idx];
  __syncthreads();
  for (int idx = tid; idx < len * V; idx += kThreads) {
    const int r = idx / V, x = idx - r * V;
    float s = 0.f;
    for (int cc = 0; cc < K; ++cc) s = fmaf(sQg[r * K + cc], hs[(size_t)cc * V + x], s);
    for (int i = 0; i <= r; ++i) s = fmaf(sQK[r * kChunk + i], sD[i * V + x], s);
    stf(o, ((int64_t)(t0 + r) * HV + j) * V + x, s);
  }
}

template <typename Tin>
cudaError_t run_prepare(const Problem &P, const Workspace &W, float *hT, cudaStream_t s) {
  cudaError_t e = launch_chunk_map(P, W, s);
  if (e != cudaSuccess) return e;
  const size_t si = intra_smem(P.K, P.V), ss = scan_smem(P.K);
  e = cudaFuncSetAttribute(simple_intra_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)si);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(simple_scan_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss);
  if (e != cudaSuccess) return e;
  if (P.NC > 0) {
    KDA_LAUNCH("simple_intra_kernel", s, simple_intra_kernel<Tin><<<dim3(P.NC, P.HV), kThreads, si, s>>>(P, W));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (P.N > 0)
    KDA_LAUNCH("simple_scan_kernel", s, simple_scan_kernel<Tin><<<dim3(P.N, P.HV, (P.V + kBV - 1) / kBV), kThreads, ss, s>>>(P, W, hT));
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t run_output(const Problem &P, const Workspace &W, void *o, cudaStream_t s) {
  if (P.NC == 0) return cudaSuccess;
  const size_t so = out_smem(P.K, P.V);
  cudaError_t e = cudaFuncSetAttribute(simple_output_kernel<Tin>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)so);
  if (e != cudaSuccess) return e;
  KDA_LAUNCH("simple_output_kernel", s, simple_output_kernel<Tin><<<dim3(P.NC, P.HV), kThreads, so, s>>>(P, W, (Tin *)o));
  return cudaGetLastError();
}

}  // namespace

cudaError_t simple_prepare(const Problem &P, const Workspace &W, float *hT, cudaStream_t s) {
  return P.bf16 ? run_prepare<__nv_bfloat16>(P, W, hT, s) : run_prepare<float>(P, W, hT, s);
}

cudaError_t simple_forward(const Problem &P, const Workspace &W, void *o, float *hT,
                           cudaStream_t s) {
  cudaError_t e = simple_prepare(P, W, hT, s);
  if (e != cudaSuccess || o == nullptr) return e;  // o NULL: the final state alone
  return P.bf16 ? run_output<__nv_bfloat16>(P, W, o, s) : run_output<float>(P, W, o, s);
}

}  // namespace kda
