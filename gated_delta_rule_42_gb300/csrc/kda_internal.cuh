// Internal definitions shared by the CUDA translation units of libkda.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder is reached through the runtime)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;    // tokens per chunk
constexpr int kMaxDim = 128;  // largest K and V the kernels are built for
// Per-slot record of the chunk tiles the states pass saves for the reverse scan
// and the gradient chain: Bk, Qg, Khat (16 KB each), Aqk, A (8 KB each), 2^G_last.
// The per-chunk record of the bf16 path (one per (chunk, value head) slot),
// written by the record kernel: swizzled bf16 operand tiles, then 2^G_last.
// Bk, Khat and A come first: the states pass reads only those 40 KB.
constexpr uint32_t kRecBK = 0;        // beta k 2^G            [64 r][128 c]
constexpr uint32_t kRecKH = 16384;    // k 2^(G_last - G)      [64 r][128 c]
constexpr uint32_t kRecAM = 32768;    // A = (I + L)^-1        [64 r][64 i]
constexpr uint32_t kRecAQK = 40960;   // Aqk                   [64 r][64 i]
constexpr uint32_t kRecQG = 49152;    // q~ 2^G                [64 r][128 c]
constexpr uint32_t kRecGAML = 65536;  // 2^G_last              fp32 [128]
constexpr uint32_t kRecStates = 40960;  // Bk | Khat | A: what the states pass loads
constexpr size_t kTileRecord = 65536 + 512;

// A chunk-table entry: the chunk's logical sequence n (-1 = unused slot), its
// first packed token, its length (1..64) and its index inside the sequence.
// A sequence entry: first packed token, length, first chunk, number of chunks.
struct Problem {
  int B, T, H, HV, K, V, N;
  int64_t Ttot;  // rows of the packed token axis (B*T)
  int NC;        // chunk-table capacity, an upper bound on the number of chunks
  bool bf16;
  bool l2norm;   // KDA_QK_L2NORM: q, k rows L2-normalised inside the op
  bool scalar_gate;  // KDA_SCALAR_GATE: g, dg are [Ttot][HV] (the fp32 kernels see g repeated over K)
  const void *q, *k, *v;
  const float *g, *beta, *h0;
  const int32_t *cu;
  const void *qr, *kr;  // the caller's raw q, k (== q, k unless the fp32 path runs on normalised copies)
};
constexpr float kL2NormEps = 1e-6f;  // epsilon of the q/k L2-norm prologue

// Device workspace, carved from the caller's buffer.  Per-(chunk, value head)
// slots are indexed slot = chunk * HV + j.
struct Workspace {
  int4 *seq;     // [N]
  int4 *chunk;   // [NC]
  int *flags;    // [0] = number of chunks, [1] = malformed-offsets flag, [2] = a bounded wait gave up,
                 // [3], [4] = (chunk, value head) slots the record / gradient kernel sent to the exact
                 // path for a wide decay span, listed in wide_rec / wide_grad; [5], [6] = slots the
                 // chunk-reference gradient / record kernel left to the block-reference one
                 // (wide_cgrad / wide_crec)
  int *wide_rec, *wide_grad;  // [NC * HV] slot lists of the fix-up launches
  int *wide_cgrad;            // [NC * HV] slots the chunk-reference gradient kernel left (flags[5])
  int *wide_crec;             // [NC * HV] slots the chunk-reference record kernel left (flags[6])
  float *G;      // [slot][64][K]   chunk-local inclusive gate cumsum
  float *Aqk;    // [slot][64][64]  lower (incl. diagonal) decayed q~ k^T
  float *A;      // [slot][64][64]  (I + L)^-1
  float *w;      // [slot][64][K]
  float *u;      // [slot][64][V]
  float *h;      // [slot][K][V]    state at chunk start
  float *delta;  // [slot][64][V]   u - w h
  // backward only
  float *dh;     // [slot][K][V]    gradient of the chunk-end state
  float *ddelta; // [slot][64][V]
  float *dqp;    // [Ttot][HV][K]   per-value-head dq~ partials
  float *dkp;    // [Ttot][HV][K]
  float *dw;     // [slot][64][K]
  // tensor-core backward (bf16, K, V = 64 or 128 in 128-wide tiles), per (chunk, value head) slot
  __nv_bfloat16 *tc_hs;     // [slot] 32 KB: chunk-start state h [K][V], swizzled operand tile (forward recompute)
  unsigned char *tc_tiles;  // [slot] kTileRecord bytes: the per-chunk record (kRec* offsets)
  unsigned char *tc_xt;     // [slot] 16 KB: swizzled X^T tile [V][64]
  unsigned char *tc_dt;     // [slot] 16 KB: swizzled D^T tile [V][64]
  __nv_bfloat16 *tc_dh;     // [slot] 32 KB: gradient of the chunk-end state [K][V], swizzled operand tile
  __nv_bfloat16 *tc_dd;     // [slot] 16 KB: gradient of the deltas [64][V], swizzled operand tile
  __nv_bfloat16 *tc_dx;     // [slot] 16 KB: dX = A^T dD [64][V], swizzled operand tile
  // fp32 path with the q/k L2-norm prologue: normalised copies of q, k (dtype, [Ttot][H][K])
  void *qn, *kn;
  // scalar gate: the gate repeated over K, and the per-channel gate gradient (fp32, [Ttot][HV][K]);
  // with the KDA gate on the fp32 path: the decay made from the raw gate, and its gradient
  float *gx, *dgx;
  // KDA gate, tensor-core backward: per-slot fp32 partials of dbias [slot][K] and dA_log [slot]
  float *gpart_b, *gpart_a;
};

// ---- the KDA gate inside the op (KDA_GATE_IN_KERNEL) ----
// With x = a + bias and s = exp(A_log): unbounded g = -s softplus(x), bounded
// (lower bound lb < 0) g = lb sigmoid(s x); g is the per-token log2 decay.
// Its parameters travel beside the Problem, to the kernels that make the decay.
struct GateArgs {
  const float *A_log, *bias;  // [HV] and [HV][K], or NULL (unit scale / no bias)
  float lb;                   // < 0: the bounded gate; 0: the unbounded one
  bool on;                    // g holds the raw gate pre-activations
};
__device__ __forceinline__ float kgate_softplus(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }
__device__ __forceinline__ float kgate_sigmoid(float y) { return 1.f / (1.f + expf(-y)); }
__device__ __forceinline__ float kgate_scale(const GateArgs &ga, int j) {
  return ga.A_log != nullptr ? expf(ga.A_log[j]) : 1.f;
}
__device__ __forceinline__ float kgate_bias(const GateArgs &ga, int K, int j, int c) {
  return ga.bias != nullptr ? ga.bias[(size_t)j * K + c] : 0.f;
}
__device__ __forceinline__ float kgate(float x, float s, float lb) {
  return lb < 0.f ? lb * kgate_sigmoid(s * x) : -s * kgate_softplus(x);
}
// (dg/dx, dg/dA_log) at x
__device__ __forceinline__ float2 kgate_grad(float x, float s, float lb) {
  if (lb < 0.f) {
    const float sg = kgate_sigmoid(s * x), t = lb * sg * (1.f - sg) * s;
    return make_float2(t, t * x);
  }
  return make_float2(-s * kgate_sigmoid(x), -s * kgate_softplus(x));
}
// The same on the hardware exponential and logarithm (the bf16 tensor-core
// path, whose results are held to bf16 accuracy; terms they drop are below
// 2^-24 of the ones they keep).
__device__ __forceinline__ float kgate_softplus_fast(float x) {
  return fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)));
}
__device__ __forceinline__ float kgate_sigmoid_fast(float y) { return __fdividef(1.f, 1.f + __expf(-y)); }
__device__ __forceinline__ float kgate_fast(float x, float s, float lb) {
  return lb < 0.f ? lb * kgate_sigmoid_fast(s * x) : -s * kgate_softplus_fast(x);
}
__device__ __forceinline__ float2 kgate_grad_fast(float x, float s, float lb) {
  if (lb < 0.f) {
    const float sg = kgate_sigmoid_fast(s * x), t = lb * sg * (1.f - sg) * s;
    return make_float2(t, t * x);
  }
  return make_float2(-s * kgate_sigmoid_fast(x), -s * kgate_softplus_fast(x));
}

// --- element access -------------------------------------------------------
__device__ __forceinline__ float ldf(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void stf(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

// TMA tensor maps of one call's per-token tensors, passed to the kernels as a
// __grid_constant__ parameter (tma.cu).  k, q: [Ttot][H][128] bf16 and v, d (a
// second per-value-head tensor: dO in the backward): [Ttot][HV][128] bf16 as
// 64 x 64 boxes with the 128-byte swizzle of the operand tiles; g:
// [Ttot][HV][128] fp32 as 64-row x 128 boxes.
struct TmaMaps {
  CUtensorMap k, q, v, g, d;
};
// Encodes the maps (v, d may be NULL: no map).  Fails without launching
// anything if the driver rejects a map (e.g. a base pointer not 16-byte aligned).
cudaError_t make_tma_maps(const Problem &P, const void *v, const void *d, TmaMaps *out);

// Number of SMs of the current device, cached per device (api.cu).
cudaError_t sm_count(int *out);

// Records the message kda_last_error() returns on the calling thread (api.cu).
void set_last_error(const char *msg);

// --- launch instrumentation (instrument.cu) -----------------------------------
void inst_begin(const char *name, cudaStream_t s);
void inst_end(cudaStream_t s);
// Wraps one kernel launch: counts it and, when timing is on, brackets it with events.
#define KDA_LAUNCH(name, stream, ...)  \
  do {                                 \
    ::kda::inst_begin(name, stream);   \
    __VA_ARGS__;                       \
    ::kda::inst_end(stream);           \
  } while (0)

// --- host-side launchers (defined in the .cu files) ---------------------------
cudaError_t launch_chunk_map(const Problem &P, const Workspace &W, cudaStream_t s);
// map + intra + scan: fills G, Aqk, A, w, u, h, delta; writes hT if not NULL
cudaError_t simple_prepare(const Problem &P, const Workspace &W, float *hT, cudaStream_t s);
cudaError_t simple_forward(const Problem &P, const Workspace &W, void *o, float *hT,
                           cudaStream_t s);
// state_only: stop after the dh scan (dh0 alone; dq .. dbeta untouched)
cudaError_t simple_backward(const Problem &P, const Workspace &W, const void *dO,
                            const float *dhT, void *dq, void *dk, void *dv, float *dg,
                            float *dbeta, float *dh0, bool state_only, cudaStream_t s);
cudaError_t launch_recurrent(const Problem &P, const GateArgs &ga, void *o, float *hT, cudaStream_t s);
// Per-chunk records (tc_prep.cu): one CTA per (chunk, value head) slot.
cudaError_t tc_prepare(const Problem &P, const GateArgs &ga, const Workspace &W, const TmaMaps &maps, int *err,
                       cudaStream_t s);
// bf16 tensor-core forward (K, V = 64 or 128): the records into W.tc_tiles (unless
// records_ready: W.tc_tiles already holds them for these q, k, g, beta), then
// the state chain.  mode is kFwdOutput (o, hT), kFwdSave (no output: per
// (chunk, value head) slot the chunk-start state and the X^T, D^T tiles go to
// W.tc_hs / tc_xt / tc_dt for the backward), both bits, or 0 (hT alone).
constexpr int kFwdOutput = 1, kFwdSave = 2;
// The chunk map and the records alone (what the reverse scan needs).
cudaError_t tc_records(const Problem &P, const GateArgs &ga, const Workspace &W, int *err, cudaStream_t s);
cudaError_t tc_forward(const Problem &P, const GateArgs &ga, const Workspace &W, void *o, float *hT, int mode,
                       bool records_ready, int *err, cudaStream_t s);
cudaError_t tc_backward_scan(const Problem &P, const Workspace &W, const void *dO, const float *dhT,
                             float *dh0, int *err, cudaStream_t s);
// Per-chunk gradients: tcgen05 products and the gradient chain in one kernel.
cudaError_t tc_backward_intra(const Problem &P, const GateArgs &ga, const Workspace &W, const void *dO, void *dv,
                              void *dq, void *dk, float *dg, float *dbeta, int *err, cudaStream_t s);
// dq = (group sum of dqp) / sqrt(K), dk = group sum of dkp, over the HV/H value heads
// q/k L2-norm prologue (l2norm.cu): normalised copies of the raw rows, and the
// partial reduction fused with the backward through the normalisation.
cudaError_t launch_l2norm_rows(const Problem &P, void *qn, void *kn, cudaStream_t s);
cudaError_t launch_group_reduce_l2norm(const Problem &P, const float *dqp, const float *dkp, void *dq, void *dk,
                                       cudaStream_t s);
// State composition for the context-parallel relay (relay.cu).
cudaError_t launch_state_compose(const float *M, const float *h, const float *c, float *out, int64_t count, int K,
                                 int V, bool transpose, cudaStream_t s);
// Scalar gate (gate.cu): [Ttot][HV] -> [Ttot][HV][K] for the kernels, and the
// per-channel gradient summed over K.
cudaError_t launch_gate_expand(const Problem &P, float *gx, cudaStream_t s);
cudaError_t launch_gate_grad_reduce(const Problem &P, const float *dgx, float *dg, cudaStream_t s);
// KDA gate (gate.cu): the fp32 path's decay from the raw gate; its backward (da
// from the per-channel dg, dA_log and dbias over the valid tokens); and the
// tensor-core path's reduction of the per-slot partials.
cudaError_t launch_kgate_apply(const Problem &P, const GateArgs &ga, float *gx, cudaStream_t s);
cudaError_t launch_kgate_grad(const Problem &P, const GateArgs &ga, const Workspace &W, const float *dgx, float *da,
                              float *dA_log, float *dbias, cudaStream_t s);
cudaError_t launch_kgate_param_reduce(const Problem &P, const Workspace &W, float *dA_log, float *dbias,
                                      cudaStream_t s);
cudaError_t launch_group_reduce(const Problem &P, const float *dqp, const float *dkp, void *dq, void *dk,
                                cudaStream_t s);
// The tensor-core kernels: bf16, K and V each 64 or 128 (a 64-wide head runs in
// the 128-wide tiles, zero-padded), and q, k, v (and a per-channel g) 16-byte
// aligned, since they arrive by TMA; other problems run the fp32 kernels.
inline bool tc_eligible(const Problem &P) {
  const uintptr_t a = (uintptr_t)P.q | (uintptr_t)P.k | (uintptr_t)P.v | (P.scalar_gate ? 0 : (uintptr_t)P.g);
  return P.bf16 && (P.K == 64 || P.K == 128) && (P.V == 64 || P.V == 128) && (a & 15) == 0;
}

}  // namespace kda
