// Scalar gate (KDA_SCALAR_GATE, the GDN variant): one log2 decay per (token,
// value head), shared by every key channel.  The fp32 chunked kernels are
// written for KDA's per-channel gate, so the scalar gate reaches them repeated
// over K (gate_expand_kernel), and the per-channel gate gradient they produce
// is summed back over K (gate_grad_reduce_kernel): dg_t = sum_c dG_t[c], the
// chain rule of g_t[c] = g_t for every c.  (The tensor-core kernels do both
// inside: they repeat the scalars into their shared-memory gate tile and sum
// dg over the channels in their dg scan.)
//
// Both kernels are HBM-bound streams: 16-byte stores of the expanded rows;
// one warp per (token, value head) row for the sum, in a fixed order.
#include "kda_internal.cuh"

namespace kda {
namespace {

// gx[(t * HV + j) * K + c] = g[t * HV + j], four channels per thread.
__global__ void __launch_bounds__(256) gate_expand_kernel(const float *__restrict__ g, float *__restrict__ gx,
                                                          int64_t rows, int K) {
  const int q4 = (K + 3) / 4;
  const int64_t total = rows * q4;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = e / q4;
    const int c = (int)(e - row * q4) * 4;
    const float x = g[row];
    float *dst = gx + row * K + c;
    if (c + 4 <= K && (K & 3) == 0) {
      *reinterpret_cast<float4 *>(dst) = make_float4(x, x, x, x);
    } else {
      for (int i = 0; i < 4 && c + i < K; ++i) dst[i] = x;
    }
  }
}

// dg[t * HV + j] = sum_c dgx[(t * HV + j) * K + c] for the tokens inside the contract.
__global__ void __launch_bounds__(256) gate_grad_reduce_kernel(Problem P, const float *__restrict__ dgx,
                                                               float *__restrict__ dg) {
  int64_t tend = P.Ttot;  // tokens at or after cu_seqlens[N] are outside the contract: not written
  if (P.cu != nullptr) {
    const int64_t e = P.cu[P.N];
    tend = e < 0 ? 0 : (e > P.Ttot ? P.Ttot : e);
  }
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= tend * P.HV) return;
  const float *src = dgx + row * P.K;
  float acc = 0.f;
  for (int c = lane; c < P.K; c += 32) acc += src[c];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) dg[row] = acc;
}

}  // namespace

cudaError_t launch_gate_expand(const Problem &P, float *gx, cudaStream_t s) {
  const int64_t rows = P.Ttot * P.HV;
  if (rows == 0) return cudaSuccess;
  int nsm = 0;
  cudaError_t e = sm_count(&nsm);
  if (e != cudaSuccess) return e;
  const int64_t total = rows * ((P.K + 3) / 4);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)nsm * 8) blocks = (int64_t)nsm * 8;
  KDA_LAUNCH("gate_expand_kernel", s, gate_expand_kernel<<<(unsigned)blocks, 256, 0, s>>>(P.g, gx, rows, P.K));
  return cudaGetLastError();
}

cudaError_t launch_gate_grad_reduce(const Problem &P, const float *dgx, float *dg, cudaStream_t s) {
  const int64_t rows = P.Ttot * P.HV;
  if (rows == 0) return cudaSuccess;
  KDA_LAUNCH("gate_grad_reduce_kernel", s, gate_grad_reduce_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(P, dgx, dg));
  return cudaGetLastError();
}

}  // namespace kda
