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
//
// The KDA gate (KDA_GATE_IN_KERNEL) reaches the fp32 kernels the same way: the
// decay made from the raw gate, and the gate's backward after them.  The
// tensor-core kernels make the decay inside their gate cumsum and leave
// per-slot partials of the parameter gradients, reduced here.
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

// ---- the KDA gate (KDA_GATE_IN_KERNEL) on the fp32 path ----

// gx = kgate(a + bias): the decay the fp32 kernels read, one element per thread step.
__global__ void __launch_bounds__(256) kgate_apply_kernel(Problem P, GateArgs ga, float *__restrict__ gx) {
  const int64_t total = P.Ttot * P.HV * P.K;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(e % P.K);
    const int j = (int)((e / P.K) % P.HV);
    gx[e] = kgate(P.g[e] + kgate_bias(ga, P.K, j, c), kgate_scale(ga, j), ga.lb);
  }
}

// One block per value head j, one thread per channel c: walks the valid tokens
// chunk by chunk in order, da = dG * dg/dx into the caller's dg, and sums
// dbias[j][c] = sum_t da and dA_log[j] = sum_{t,c} dG * dg/dA_log in a fixed
// order (in fp64 on this fp32 path, whose results are held to fp32 accuracy).
__global__ void __launch_bounds__(128) kgate_grad_kernel(Problem P, GateArgs ga, Workspace W, const float *__restrict__ dgx,
                                                         float *__restrict__ da, float *__restrict__ dA_log,
                                                         float *__restrict__ dbias) {
  __shared__ double red[128];
  const int j = blockIdx.x, c = threadIdx.x;
  double pb = 0.0, pa = 0.0;  // fp64 partial sums: these reduce over every valid token
  if (c < P.K) {
    const float s = kgate_scale(ga, j), b = kgate_bias(ga, P.K, j, c);
    for (int ci = 0; ci < P.NC; ++ci) {
      const int4 ch = W.chunk[ci];
      if (ch.x < 0) break;  // the valid chunks come first
      for (int r = 0; r < ch.z; ++r) {
        const size_t e = ((size_t)(ch.y + r) * P.HV + j) * P.K + c;
        const float2 d = kgate_grad(P.g[e] + b, s, ga.lb);
        const float v = dgx[e];
        da[e] = v * d.x;
        pb += (double)(v * d.x);
        pa += (double)v * (double)d.y;
      }
    }
    if (dbias != nullptr) dbias[(size_t)j * P.K + c] = (float)pb;
  }
  red[c] = pa;
  __syncthreads();
  if (c == 0 && dA_log != nullptr) {
    double t = 0.0;
    for (int i = 0; i < P.K; ++i) t += red[i];
    dA_log[j] = (float)t;
  }
}

// Tensor-core path: dbias[j][c] and dA_log[j] from the per-slot partials the
// gradient kernel left (slot = chunk * HV + j, rows 128 wide), summed over the
// valid chunks in a fixed order.  Block (j, 32 channels): warp w sums the
// chunks w, w + 8, ..., then the 8 warp sums are added in order; block y = 0
// also sums the dA_log partials the same way over its 256 threads.
__global__ void __launch_bounds__(256) kgate_param_reduce_kernel(Problem P, Workspace W, float *__restrict__ dA_log,
                                                                 float *__restrict__ dbias) {
  __shared__ float part[8][32];
  __shared__ float pa_s[256];
  const int j = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5, c = blockIdx.y * 32 + lane;
  const int nch = *(volatile const int *)W.flags;  // chunks mapped: the valid chunks come first
  float pb = 0.f;
  for (int ci = w; ci < nch; ci += 8) pb += W.gpart_b[((size_t)ci * P.HV + j) * kMaxDim + c];
  part[w][lane] = pb;
  float pa = 0.f;
  if (blockIdx.y == 0)
    for (int ci = threadIdx.x; ci < nch; ci += 256) pa += W.gpart_a[(size_t)ci * P.HV + j];
  pa_s[threadIdx.x] = pa;
  __syncthreads();
  if (w == 0 && c < P.K && dbias != nullptr) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += part[i][lane];
    dbias[(size_t)j * P.K + c] = t;
  }
  if (blockIdx.y == 0 && threadIdx.x == 32 && dA_log != nullptr) {
    float t = 0.f;
    for (int i = 0; i < 256; ++i) t += pa_s[i];
    dA_log[j] = t;
  }
}

}  // namespace

cudaError_t launch_kgate_apply(const Problem &P, const GateArgs &ga, float *gx, cudaStream_t s) {
  const int64_t total = P.Ttot * P.HV * P.K;
  if (total == 0) return cudaSuccess;
  int nsm = 0;
  cudaError_t e = sm_count(&nsm);
  if (e != cudaSuccess) return e;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)nsm * 8) blocks = (int64_t)nsm * 8;
  KDA_LAUNCH("kgate_apply_kernel", s, kgate_apply_kernel<<<(unsigned)blocks, 256, 0, s>>>(P, ga, gx));
  return cudaGetLastError();
}

cudaError_t launch_kgate_grad(const Problem &P, const GateArgs &ga, const Workspace &W, const float *dgx, float *da,
                              float *dA_log, float *dbias, cudaStream_t s) {
  if (P.NC == 0) return cudaSuccess;
  KDA_LAUNCH("kgate_grad_kernel", s, kgate_grad_kernel<<<P.HV, 128, 0, s>>>(P, ga, W, dgx, da, dA_log, dbias));
  return cudaGetLastError();
}

cudaError_t launch_kgate_param_reduce(const Problem &P, const Workspace &W, float *dA_log, float *dbias,
                                      cudaStream_t s) {
  if ((dA_log == nullptr && dbias == nullptr) || P.NC == 0) return cudaSuccess;
  KDA_LAUNCH("kgate_param_reduce_kernel", s,
             kgate_param_reduce_kernel<<<dim3(P.HV, (P.K + 31) / 32), 256, 0, s>>>(P, W, dA_log, dbias));
  return cudaGetLastError();
}

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
