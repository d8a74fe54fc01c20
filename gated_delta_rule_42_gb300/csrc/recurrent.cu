// Token-by-token recurrent KDA forward (inference).
//
// One block per (sequence, value head, 32 value columns); a lane pair holds
// one column of the fp32 state S[K][.] in registers (half the channels each,
// combined with one shuffle) and walks the
// sequence's tokens in order, computing in fp32 whatever the input dtype --
// the shape of the recurrent_kda kernel described in "kda in torchtitan
// (training)" (pytorch/torchtitan PR #4164, agent note: state [K, BV] in
// registers, one program per (sequence, head, value block)).
//
// Per token: S <- diag(2^g) S ; e = S^T k ; S <- S + k (beta (v - e))^T ;
// o = S^T q / sqrt(K).  An empty slot leaves the state untouched.  With the
// q/k L2-norm prologue, k and q are divided by their row norms (sqrt of the sum
// of squares + eps), applied as the factors rk and rq.  A scalar gate (one
// decay per token and value head) is read as such.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kCols = 32;            // value columns per block
constexpr int kThreadsR = 2 * kCols; // a lane pair holds one column (half the channels each)

template <typename Tin, int KHALF>
__global__ void __launch_bounds__(kThreadsR)
recurrent_kernel(Problem P, GateArgs ga, Tin *__restrict__ o, float *__restrict__ hT) {
  const int n = blockIdx.x, j = blockIdx.y;
  const int half = threadIdx.x & 1, x = blockIdx.z * kCols + (threadIdx.x >> 1);
  const int K = P.K, V = P.V, HV = P.HV, H = P.H, h = j / (HV / H);
  const Tin *q = (const Tin *)P.q, *k = (const Tin *)P.k, *v = (const Tin *)P.v;
  const float scale = 1.0f / sqrtf((float)K);
  const bool active = x < V;
  const size_t base = ((size_t)n * HV + j) * K * V;
  const int c0 = half * KHALF;  // this lane's channels: c0 .. c0 + KHALF - 1

  __shared__ float sk[2 * KHALF], sq[2 * KHALF], sa[2 * KHALF];
  float S[KHALF];
#pragma unroll
  for (int c = 0; c < KHALF; ++c)
    S[c] = (c0 + c < K && active && P.h0 != nullptr) ? P.h0[base + (size_t)(c0 + c) * V + x] : 0.f;

  int64_t t0, t1;
  if (P.cu != nullptr) {
    t0 = P.cu[n];
    t1 = P.cu[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > P.Ttot) t1 = t0;  // malformed offsets: no tokens
  } else {
    t0 = (int64_t)n * P.T;
    t1 = t0 + P.T;
  }
  for (int64_t t = t0; t < t1; ++t) {
    __syncthreads();
    for (int c = threadIdx.x; c < 2 * KHALF; c += kThreadsR) {
      float kv = 0.f, qv = 0.f, av = 1.f;
      if (c < K) {
        const int64_t e = (t * H + h) * K + c;
        kv = ldf(k, e);
        qv = ldf(q, e);
        const float gv = P.scalar_gate ? P.g[t * HV + j] : P.g[(t * HV + j) * K + c];
        // the KDA gate inside the op: the decay from the raw gate
        av = exp2f(ga.on ? kgate(gv + kgate_bias(ga, K, j, c), kgate_scale(ga, j), ga.lb) : gv);
      }
      sk[c] = kv;
      sq[c] = qv;
      sa[c] = av;
    }
    const float b = P.beta[t * HV + j];
    __syncthreads();
    float rk = 1.f, rq = scale;  // key and query row factors
    if (P.l2norm) {  // q/k L2-norm prologue: every thread sums the two rows itself
      float a2 = 0.f, b2 = 0.f;
      for (int c = 0; c < K; ++c) {
        a2 = fmaf(sk[c], sk[c], a2);
        b2 = fmaf(sq[c], sq[c], b2);
      }
      rk = 1.0f / sqrtf(a2 + kL2NormEps);
      rq = scale / sqrtf(b2 + kL2NormEps);
    }
    float e = 0.f;
#pragma unroll
    for (int c = 0; c < KHALF; ++c) {
      S[c] *= sa[c0 + c];
      e = fmaf(S[c], sk[c0 + c], e);
    }
    e += __shfl_xor_sync(0xffffffffu, e, 1);
    const float d = active ? b * (ldf(v, (t * HV + j) * V + x) - e * rk) * rk : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < KHALF; ++c) {
      S[c] = fmaf(sk[c0 + c], d, S[c]);
      acc = fmaf(S[c], sq[c0 + c], acc);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (active && half == 0) stf(o, (t * HV + j) * V + x, acc * rq);
  }
  if (hT != nullptr && active) {
#pragma unroll
    for (int c = 0; c < KHALF; ++c)
      if (c0 + c < K) hT[base + (size_t)(c0 + c) * V + x] = S[c];
  }
}

template <typename Tin>
cudaError_t run(const Problem &P, const GateArgs &ga, void *o, float *hT, cudaStream_t s) {
  if (P.N == 0) return cudaSuccess;
  const dim3 grid(P.N, P.HV, (P.V + kCols - 1) / kCols);
  if (P.K <= 64)
    KDA_LAUNCH("recurrent_kernel", s, recurrent_kernel<Tin, 32><<<grid, kThreadsR, 0, s>>>(P, ga, (Tin *)o, hT));
  else
    KDA_LAUNCH("recurrent_kernel", s, recurrent_kernel<Tin, 64><<<grid, kThreadsR, 0, s>>>(P, ga, (Tin *)o, hT));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const Problem &P, const GateArgs &ga, void *o, float *hT, cudaStream_t s) {
  return P.bf16 ? run<__nv_bfloat16>(P, ga, o, hT, s) : run<float>(P, ga, o, hT, s);
}

}  // namespace kda
