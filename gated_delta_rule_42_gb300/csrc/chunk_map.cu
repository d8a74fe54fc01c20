// Device-side chunk map: from the packed offsets (or a dense B x T batch) to
// the list of 64-token chunks.  Chunks never straddle a sequence boundary and
// an empty slot (repeated offset) produces no chunk.  Runs entirely on the
// device, so a CUDA graph can be replayed with new offsets (the
// "CUDA-graph replay with mutated boundaries" check of the recurrent_kda test
// plan in "kda in torchtitan (training)", pytorch/torchtitan PR #4164).
//
// Malformed offsets (decreasing, negative, past the token axis) are treated
// as empty sequences and flagged in flags[1]; chunk indices are clamped to the
// table capacity, so no later kernel can address memory outside its buffers.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kMapThreads = 1024;

__global__ void __launch_bounds__(kMapThreads)
chunk_map_kernel(const int32_t *__restrict__ cu, int B, int T, int N, int64_t Ttot, int NC,
                 int4 *__restrict__ seq, int4 *__restrict__ chunk, int *__restrict__ flags) {
  __shared__ int s_scan[kMapThreads];
  __shared__ int s_carry;
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_carry = 0;
    s_bad = 0;
    flags[2] = 0;  // the call's bounded-wait error word: every call starts clean
    flags[3] = 0;  // and its counts of slots on the exact (wide-decay) path
    flags[4] = 0;
    flags[5] = 0;  // and on the block-reference path (wide chunk span)
    flags[6] = 0;
  }
  __syncthreads();
  for (int base = 0; base < N; base += kMapThreads) {
    const int n = base + tid;
    int t0 = 0, len = 0, nch = 0;
    if (n < N) {
      if (cu != nullptr) {
        const int a = cu[n], b = cu[n + 1];
        if (a < 0 || b < a || (int64_t)b > Ttot) {
          s_bad = 1;  // benign race: every writer stores 1
        } else {
          t0 = a;
          len = b - a;
        }
      } else {
        t0 = n * T;
        len = T;
      }
      nch = (len + kChunk - 1) / kChunk;
    }
    s_scan[tid] = nch;
    __syncthreads();
    for (int off = 1; off < kMapThreads; off <<= 1) {
      const int x = tid >= off ? s_scan[tid - off] : 0;
      __syncthreads();
      s_scan[tid] += x;
      __syncthreads();
    }
    int first = s_carry + s_scan[tid] - nch;
    if (n < N) {
      if (first >= NC) {
        if (nch > 0) s_bad = 1;
        first = NC;
        nch = 0;
      } else if (first + nch > NC) {
        nch = NC - first;
        s_bad = 1;
      }
      seq[n] = make_int4(t0, len, first, nch);
      for (int c = 0; c < nch; ++c) {
        const int rem = len - c * kChunk;
        chunk[first + c] = make_int4(n, t0 + c * kChunk, rem < kChunk ? rem : kChunk, c);
      }
    }
    __syncthreads();
    if (tid == kMapThreads - 1) s_carry += s_scan[tid];
    __syncthreads();
  }
  const int total = s_carry < NC ? s_carry : NC;
  for (int c = total + tid; c < NC; c += kMapThreads) chunk[c] = make_int4(-1, 0, 0, 0);
  if (tid == 0) {
    flags[0] = total;
    flags[1] = s_bad;
  }
}

}  // namespace

cudaError_t launch_chunk_map(const Problem &P, const Workspace &W, cudaStream_t s) {
  KDA_LAUNCH("chunk_map_kernel", s, chunk_map_kernel<<<1, kMapThreads, 0, s>>>(P.cu, P.B, P.T, P.N, P.Ttot, P.NC, W.seq, W.chunk,
                                             W.flags));
  return cudaGetLastError();
}

}  // namespace kda
