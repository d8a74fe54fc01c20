// State composition for the context-parallel state relay.
//
// When a sequence is split across ranks, rank r sees its segment as an affine
// map of the state it starts from: S_end = M_r S_start + c_r, with c_r its final
// state from a zero start and M_r (K x K) the product of the segment's per-token
// transitions diag(2^g_t) - beta_t k_t k_t^T diag(2^g_t), the linear part of the
// delta rule.  An exclusive scan of these maps across ranks gives every rank its
// true start state -- the state relay of synchronous context parallelism in
// "[KDA] Add Paddle training compatibility" (PFCCLab/flash-linear-attention
// PR #2, context-parallel test plan) -- and the backward runs it in reverse with
// M_r^T on the state gradients.
//
// out[i] = op(M[i]) h[i] + c[i] for every (sequence, value head) i, fp32,
// op = identity or transpose; one CTA per (i, 8-row block of out) -- enough
// CTAs to spread the few states of a relay step over the SMs -- each thread one
// output column, K streamed through shared memory.  Each output is
// a fixed-order sum, so the result does not depend on the launch.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kRows = 8;  // output rows per CTA

__global__ void __launch_bounds__(128)
state_compose_kernel(const float *__restrict__ M, const float *__restrict__ h, const float *__restrict__ c,
                     float *__restrict__ out, int K, int V, int transpose) {
  __shared__ float mrow[kRows][kMaxDim + 1];
  const int64_t i = blockIdx.x;
  const int a0 = blockIdx.y * kRows;
  const float *Mi = M + i * K * K;
  const float *hi = h + i * K * V;
  for (int e = threadIdx.x; e < kRows * K; e += blockDim.x) {
    const int ar = e / K, b = e - ar * K, a = a0 + ar;
    mrow[ar][b] = a < K ? (transpose ? Mi[(int64_t)b * K + a] : Mi[(int64_t)a * K + b]) : 0.f;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < V; x += blockDim.x) {
    float acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[r] = 0.f;
#pragma unroll 8
    for (int b = 0; b < K; ++b) {
      const float hb = hi[(int64_t)b * V + x];
#pragma unroll
      for (int r = 0; r < kRows; ++r) acc[r] = fmaf(mrow[r][b], hb, acc[r]);
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int a = a0 + r;
      if (a < K) {
        const int64_t o = (i * K + a) * V + x;
        out[o] = acc[r] + (c != nullptr ? c[o] : 0.f);
      }
    }
  }
}

}  // namespace

cudaError_t launch_state_compose(const float *M, const float *h, const float *c, float *out, int64_t count, int K,
                                 int V, bool transpose, cudaStream_t s) {
  if (count == 0) return cudaSuccess;
  const dim3 grid((unsigned)count, (unsigned)((K + kRows - 1) / kRows));
  KDA_LAUNCH("state_compose_kernel", s, state_compose_kernel<<<grid, 128, 0, s>>>(M, h, c, out, K, V, transpose ? 1 : 0));
  return cudaGetLastError();
}

}  // namespace kda
