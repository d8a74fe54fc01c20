// q/k L2-norm prologue (KDA_QK_L2NORM): each (token, head) row of q and k is
// divided by sqrt(sum of its squares + eps) over the K channels, and the
// backward carries the row gradients through it:
//   y = x r,  r = (sum_c x_c^2 + eps)^(-1/2);   dx = r (dy - y (y . dy)).
// The KDA layer of "kda in torchtitan (training)" (pytorch/torchtitan PR #4164)
// imports an `l2norm` beside `recurrent_kda`; the pages print neither formula
// nor epsilon, so eps = 1e-6 is this library's choice.
//
// The bf16 tensor-core path normalises inside its tile passes (the record
// kernel and the per-chunk gradient kernel read raw q, k anyway), so its only
// extra kernel is the backward below, fused with the sum of the per-value-head
// dq, dk partials.  The fp32 path normalises into workspace copies first.
// One warp per row (K <= 128: at most four channels per lane), reductions by
// warp shuffles in a fixed order.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row

template <typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
l2norm_rows_kernel(const T *__restrict__ q, const T *__restrict__ k, T *__restrict__ qn, T *__restrict__ kn,
                   int64_t rows, int K) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  for (int which = 0; which < 2; ++which) {
    const T *x = (which ? k : q) + row * K;
    T *y = (which ? kn : qn) + row * K;
    float v[4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      v[i] = c < K ? ldf(x, c) : 0.f;
      ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss + kL2NormEps);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      if (c < K) stf(y, c, v[i] * r);
    }
  }
}

// dq, dk of the raw rows: the per-value-head partials of dq~ and dk (fp32,
// [Ttot][HV][K]) summed over the HV / H value heads of each q/k head (dq~ times
// the 1/sqrt(K) query scale), then carried through the row normalisation.
template <typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
group_reduce_l2norm_kernel(Problem P, const float *__restrict__ dqp, const float *__restrict__ dkp,
                           T *__restrict__ dq, T *__restrict__ dk) {
  const int lane = threadIdx.x & 31;
  const int H = P.H, HV = P.HV, K = P.K, rr = HV / H;
  int64_t tend = P.Ttot;  // tokens at or after cu_seqlens[N] are outside the contract: not written
  if (P.cu != nullptr) {
    const int64_t e = P.cu[P.N];
    tend = e < 0 ? 0 : (e > P.Ttot ? P.Ttot : e);
  }
  const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= tend * H) return;
  const int64_t t = row / H;
  const int h = (int)(row - t * H);
  const float qscale = 1.0f / sqrtf((float)K);
  for (int which = 0; which < 2; ++which) {
    const T *x = (const T *)(which ? P.kr : P.qr) + row * K;
    const float *part = which ? dkp : dqp;
    const float sc = which ? 1.f : qscale;
    float v[4], d[4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      v[i] = 0.f;
      d[i] = 0.f;
      if (c < K) {
        v[i] = ldf(x, c);
        float acc = 0.f;
        for (int jj = 0; jj < rr; ++jj) acc += part[(t * HV + (int64_t)h * rr + jj) * K + c];
        d[i] = acc * sc;
      }
      ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss + kL2NormEps);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) dot = fmaf(v[i] * r, d[i], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    T *out = (which ? dk : dq) + row * K;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      if (c < K) stf(out, c, r * (d[i] - v[i] * r * dot));
    }
  }
}

// The same for K = 128 (the bf16 tensor-core path): lane = four consecutive
// channels, so every load and store is one vector access, and the q and k rows
// of a (token, head) are processed together to keep more loads in flight.
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}
__device__ __forceinline__ void ld4(const float *p, float (&x)[4]) {
  const float4 u = *reinterpret_cast<const float4 *>(p);
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float (&x)[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
}
__device__ __forceinline__ void st4(float *p, const float (&x)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}

template <typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
group_reduce_l2norm128_kernel(Problem P, const float *__restrict__ dqp, const float *__restrict__ dkp,
                              T *__restrict__ dq, T *__restrict__ dk) {
  constexpr int K = 128;
  const int lane = threadIdx.x & 31;
  const int H = P.H, HV = P.HV, rr = HV / H;
  int64_t tend = P.Ttot;  // tokens at or after cu_seqlens[N] are outside the contract: not written
  if (P.cu != nullptr) {
    const int64_t e = P.cu[P.N];
    tend = e < 0 ? 0 : (e > P.Ttot ? P.Ttot : e);
  }
  const int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= tend * H) return;
  const int64_t t = row / H;
  const int h = (int)(row - t * H);
  const int c = 4 * lane;
  float xq[4], xk[4], dq4[4] = {0.f, 0.f, 0.f, 0.f}, dk4[4] = {0.f, 0.f, 0.f, 0.f};
  ld4((const T *)P.qr + row * K + c, xq);
  ld4((const T *)P.kr + row * K + c, xk);
  for (int jj = 0; jj < rr; ++jj) {
    const int64_t pi = (t * HV + (int64_t)h * rr + jj) * K + c;
    float a[4], b[4];
    ld4(dqp + pi, a);
    ld4(dkp + pi, b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      dq4[e] += a[e];
      dk4[e] += b[e];
    }
  }
  const float qscale = 0.08838834764831845f;  // 1/sqrt(128)
  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    dq4[e] *= qscale;
    sq = fmaf(xq[e], xq[e], sq);
    sk = fmaf(xk[e], xk[e], sk);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, o);
    sk += __shfl_xor_sync(0xffffffffu, sk, o);
  }
  const float rq = 1.0f / sqrtf(sq + kL2NormEps), rk = 1.0f / sqrtf(sk + kL2NormEps);
  float pq = 0.f, pk = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    pq = fmaf(xq[e] * rq, dq4[e], pq);
    pk = fmaf(xk[e] * rk, dk4[e], pk);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pq += __shfl_xor_sync(0xffffffffu, pq, o);
    pk += __shfl_xor_sync(0xffffffffu, pk, o);
  }
  float oq[4], ok[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    oq[e] = rq * (dq4[e] - xq[e] * rq * pq);
    ok[e] = rk * (dk4[e] - xk[e] * rk * pk);
  }
  st4(dq + row * K + c, oq);
  st4(dk + row * K + c, ok);
}

}  // namespace

cudaError_t launch_l2norm_rows(const Problem &P, void *qn, void *kn, cudaStream_t s) {
  const int64_t rows = P.Ttot * P.H;
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
  if (P.bf16)
    KDA_LAUNCH("l2norm_rows_kernel", s, l2norm_rows_kernel<__nv_bfloat16><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
        (const __nv_bfloat16 *)P.qr, (const __nv_bfloat16 *)P.kr, (__nv_bfloat16 *)qn, (__nv_bfloat16 *)kn, rows, P.K));
  else
    KDA_LAUNCH("l2norm_rows_kernel", s, l2norm_rows_kernel<float><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
        (const float *)P.qr, (const float *)P.kr, (float *)qn, (float *)kn, rows, P.K));
  return cudaGetLastError();
}

cudaError_t launch_group_reduce_l2norm(const Problem &P, const float *dqp, const float *dkp, void *dq, void *dk,
                                       cudaStream_t s) {
  const int64_t rows = P.Ttot * P.H;
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
  // the vector kernel needs 16-byte aligned rows of q, k, dq and dk
  const bool vec = P.K == 128 && (((uintptr_t)P.qr | (uintptr_t)P.kr | (uintptr_t)dq | (uintptr_t)dk) & 15) == 0;
  if (vec && P.bf16)
    KDA_LAUNCH("group_reduce_l2norm_kernel", s, group_reduce_l2norm128_kernel<__nv_bfloat16><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
        P, dqp, dkp, (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk));
  else if (vec)
    KDA_LAUNCH("group_reduce_l2norm_kernel", s, group_reduce_l2norm128_kernel<float><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
        P, dqp, dkp, (float *)dq, (float *)dk));
  else if (P.bf16)
    KDA_LAUNCH("group_reduce_l2norm_kernel", s, group_reduce_l2norm_kernel<__nv_bfloat16><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
        P, dqp, dkp, (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk));
  else
    KDA_LAUNCH("group_reduce_l2norm_kernel", s, group_reduce_l2norm_kernel<float><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
        P, dqp, dkp, (float *)dq, (float *)dk));
  return cudaGetLastError();
}

}  // namespace kda
