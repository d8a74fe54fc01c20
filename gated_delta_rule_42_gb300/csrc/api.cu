// C ABI of libkda: argument validation, workspace layout and dispatch.
#include <atomic>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

thread_local char g_err[512] = "";

kda_status fail(kda_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

kda_status cuda_fail(cudaError_t e, const char *where) {
  return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Checks every host-visible property of the problem and fills P.
kda_status validate(const kda_inputs *in, Problem &P) {
  if (in == nullptr) return fail(KDA_ERR_INVALID_ARG, "inputs is NULL");
  if (in->B < 1 || in->T < 0 || in->H < 1 || in->HV < 1 || in->K < 1 || in->V < 1)
    return fail(KDA_ERR_INVALID_ARG, "sizes must be positive (B=%d T=%d H=%d HV=%d K=%d V=%d)",
                in->B, in->T, in->H, in->HV, in->K, in->V);
  if (in->HV % in->H != 0)
    return fail(KDA_ERR_INVALID_ARG, "HV (%d) must be a multiple of H (%d)", in->HV, in->H);
  if (in->K > kMaxDim || in->V > kMaxDim)
    return fail(KDA_ERR_UNSUPPORTED, "K=%d V=%d: head dims above %d are not implemented", in->K,
                in->V, kMaxDim);
  if (in->HV > 65535) return fail(KDA_ERR_UNSUPPORTED, "HV=%d above 65535", in->HV);
  if (in->dtype != KDA_F32 && in->dtype != KDA_BF16)
    return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)in->dtype);
  if ((in->flags & ~(int)(KDA_QK_L2NORM | KDA_SCALAR_GATE | KDA_GATE_IN_KERNEL)) != 0)
    return fail(KDA_ERR_INVALID_ARG, "unknown flags 0x%x", (unsigned)in->flags);
  if ((in->flags & KDA_GATE_IN_KERNEL) != 0) {
    if (in->gate == nullptr) return fail(KDA_ERR_INVALID_ARG, "KDA_GATE_IN_KERNEL needs gate parameters");
    if ((in->flags & KDA_SCALAR_GATE) != 0)
      return fail(KDA_ERR_UNSUPPORTED, "KDA_GATE_IN_KERNEL is not combined with KDA_SCALAR_GATE");
    const float lb = in->gate->lower_bound;
    if (!(lb <= 0.f) || lb < -3.0e38f) return fail(KDA_ERR_INVALID_ARG, "gate lower_bound must be finite and <= 0");
  }
  const int64_t Ttot = (int64_t)in->B * in->T;
  if (Ttot * (in->HV > in->H ? in->HV : in->H) * kMaxDim >= ((int64_t)1 << 46))
    return fail(KDA_ERR_UNSUPPORTED, "problem too large");
  if (in->cu_seqlens != nullptr) {
    if (in->B != 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens requires B == 1 (B=%d)", in->B);
    if (in->N < 0) return fail(KDA_ERR_INVALID_ARG, "N=%d must be >= 0", in->N);
  } else if (in->N != in->B) {
    return fail(KDA_ERR_INVALID_ARG, "dense batch: N (%d) must equal B (%d)", in->N, in->B);
  }
  if (in->N > (1 << 24)) return fail(KDA_ERR_UNSUPPORTED, "N=%d too large", in->N);
  if (Ttot > 0 && (in->q == nullptr || in->k == nullptr || in->v == nullptr ||
                   in->g == nullptr || in->beta == nullptr))
    return fail(KDA_ERR_INVALID_ARG, "q, k, v, g and beta are required");
  P.B = in->B;
  P.T = in->T;
  P.H = in->H;
  P.HV = in->HV;
  P.K = in->K;
  P.V = in->V;
  P.N = in->N;
  P.Ttot = Ttot;
  const int64_t per = ((int64_t)in->T + kChunk - 1) / kChunk;
  const int64_t nc = in->cu_seqlens != nullptr ? per + in->N : per * in->B;
  if (nc >= (1 << 30)) return fail(KDA_ERR_UNSUPPORTED, "too many chunks");
  P.NC = (int)nc;
  P.bf16 = in->dtype == KDA_BF16;
  P.l2norm = (in->flags & KDA_QK_L2NORM) != 0;
  P.scalar_gate = (in->flags & KDA_SCALAR_GATE) != 0;
  P.q = in->q;
  P.k = in->k;
  P.qr = in->q;
  P.kr = in->k;
  P.v = in->v;
  P.g = in->g;
  P.beta = in->beta;
  P.h0 = in->h0;
  P.cu = in->cu_seqlens;
  return KDA_OK;
}

bool use_tc(const Problem &P) { return tc_eligible(P); }

// The KDA gate's parameters of a validated call (on == false without KDA_GATE_IN_KERNEL).
GateArgs gate_args(const kda_inputs *in) {
  GateArgs ga{nullptr, nullptr, 0.f, false};
  if ((in->flags & KDA_GATE_IN_KERNEL) != 0) ga = GateArgs{in->gate->A_log, in->gate->bias, in->gate->lower_bound, true};
  return ga;
}

// The forward context of the tensor-core path: what a forward keeps for its
// backward -- the per-chunk records and, per (chunk, value head) slot, the
// chunk-start state and the X^T, D^T tiles -- so that the backward runs
// neither the record kernel nor the states pass.  Returns its size (0 on the
// general path, which keeps nothing); with base != NULL also points W's
// tc_tiles, tc_hs, tc_xt and tc_dt into it.
size_t ctx_layout(const Problem &P, char *base, Workspace *W) {
  if (!use_tc(P)) return 0;
  const size_t slots = (size_t)P.NC * P.HV;
  const size_t rec = align256(kTileRecord * slots), hs = align256(2 * slots * kMaxDim * kMaxDim);
  const size_t t16 = align256(16384 * slots);
  if (base != nullptr && W != nullptr) {
    W->tc_tiles = (unsigned char *)base;
    W->tc_hs = (__nv_bfloat16 *)(base + rec);
    W->tc_xt = (unsigned char *)(base + rec + hs);
    W->tc_dt = (unsigned char *)(base + rec + hs + t16);
  }
  return rec + hs + 2 * t16;
}

// Workspace regions, in order.  Returns the total size; with base != NULL
// also fills W.  With with_ctx the regions the forward context holds are
// left out (ctx_layout points W at them).
size_t layout(const Problem &P, bool kgate, bool backward, bool with_ctx, char *base, Workspace *W) {
  const size_t slots = (size_t)P.NC * P.HV;
  const size_t K = P.K, V = P.V, C = kChunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return base ? (void *)(base + at) : nullptr;
  };
  Workspace w;
  memset(&w, 0, sizeof(w));
  w.seq = (int4 *)take(sizeof(int4) * (size_t)(P.N > 0 ? P.N : 1));
  w.chunk = (int4 *)take(sizeof(int4) * (size_t)(P.NC > 0 ? P.NC : 1));
  w.flags = (int *)take(sizeof(int) * 8);
  if (use_tc(P)) {  // slots the record / gradient kernel leaves to its exact-path fix-up launch
    w.wide_rec = (int *)take(sizeof(int) * (slots > 0 ? slots : 1));
    w.wide_crec = (int *)take(sizeof(int) * (slots > 0 ? slots : 1));
    if (backward) {
      w.wide_grad = (int *)take(sizeof(int) * (slots > 0 ? slots : 1));
      w.wide_cgrad = (int *)take(sizeof(int) * (slots > 0 ? slots : 1));
    }
  }
  if ((P.scalar_gate || kgate) && !use_tc(P)) {  // fp32 path: the decay per channel (and its gradient)
    w.gx = (float *)take(sizeof(float) * (size_t)P.Ttot * P.HV * K);
    if (backward) w.dgx = (float *)take(sizeof(float) * (size_t)P.Ttot * P.HV * K);
  }
  if (kgate && use_tc(P) && backward) {  // per-slot fp32 partials of the gate's parameter gradients
    w.gpart_b = (float *)take(sizeof(float) * slots * kMaxDim);
    w.gpart_a = (float *)take(sizeof(float) * slots);
  }
  if (use_tc(P)) {
    if (!with_ctx) w.tc_tiles = (unsigned char *)take(kTileRecord * slots);  // per-chunk records of the preparation kernel
    if (backward) {  // tensor-core backward: per-slot tiles passed between its kernels
      if (!with_ctx) {
        w.tc_hs = (__nv_bfloat16 *)take(2 * slots * kMaxDim * kMaxDim);
        w.tc_xt = (unsigned char *)take(16384 * slots);
        w.tc_dt = (unsigned char *)take(16384 * slots);
      }
      w.tc_dh = (__nv_bfloat16 *)take(2 * slots * kMaxDim * kMaxDim);  // 128-wide tiles (a 64-wide head padded)
      w.tc_dd = (__nv_bfloat16 *)take(2 * slots * C * kMaxDim);
      w.tc_dx = (__nv_bfloat16 *)take(2 * slots * C * kMaxDim);
      if (P.HV != P.H) {  // fp32 dq, dk partials, reduced (and normalised) per q/k head afterwards
        w.dqp = (float *)take(sizeof(float) * (size_t)P.Ttot * P.HV * K);
        w.dkp = (float *)take(sizeof(float) * (size_t)P.Ttot * P.HV * K);
      }
    }
    if (W) *W = w;
    return off;
  }
  if (P.l2norm) {  // normalised copies of q, k for the fp32 path
    const size_t e = P.bf16 ? 2 : 4;
    w.qn = take(e * (size_t)P.Ttot * P.H * K);
    w.kn = take(e * (size_t)P.Ttot * P.H * K);
  }
  w.G = (float *)take(sizeof(float) * slots * C * K);
  w.Aqk = (float *)take(sizeof(float) * slots * C * C);
  w.A = (float *)take(sizeof(float) * slots * C * C);
  w.w = (float *)take(sizeof(float) * slots * C * K);
  w.u = (float *)take(sizeof(float) * slots * C * V);
  w.h = (float *)take(sizeof(float) * slots * K * V);
  w.delta = (float *)take(sizeof(float) * slots * C * V);
  if (backward) {
    w.dh = (float *)take(sizeof(float) * slots * K * V);
    w.ddelta = (float *)take(sizeof(float) * slots * C * V);
    w.dqp = (float *)take(sizeof(float) * (size_t)P.Ttot * P.HV * K);
    w.dkp = (float *)take(sizeof(float) * (size_t)P.Ttot * P.HV * K);
    w.dw = (float *)take(sizeof(float) * slots * C * K);
  }
  if (W) *W = w;
  return off;
}

// With a scalar gate the fp32 chunked kernels read the gate repeated over K
// from the workspace; the tensor-core kernels and the recurrent kernel read
// the scalars directly.
// With the KDA gate the fp32 kernels read the decay made from the raw gate; the
// tensor-core kernels make it themselves.
cudaError_t gate_per_channel(const Problem &P, const GateArgs &ga, const Workspace &W, Problem *Pg, cudaStream_t s) {
  if ((!P.scalar_gate && !ga.on) || use_tc(P)) return cudaSuccess;
  cudaError_t e = ga.on ? launch_kgate_apply(P, ga, W.gx, s) : launch_gate_expand(P, W.gx, s);
  Pg->g = W.gx;
  return e;
}

// The fp32 path with the q/k L2-norm prologue runs on normalised copies of q
// and k in the workspace; the raw rows stay in qr, kr for the backward.
cudaError_t normalised_copies(const Problem &P, const Workspace &W, Problem *Pn, cudaStream_t s) {
  if (!P.l2norm) return cudaSuccess;
  cudaError_t e = launch_l2norm_rows(P, W.qn, W.kn, s);
  Pn->q = W.qn;
  Pn->k = W.kn;
  return e;
}

kda_status check_ws(size_t need, const void *ws, size_t bytes, const char *what = "workspace") {
  if (need == 0) return KDA_OK;
  if (ws == nullptr) return fail(KDA_ERR_WORKSPACE, "%s is NULL (%zu bytes needed)", what, need);
  if (bytes < need)
    return fail(KDA_ERR_WORKSPACE, "%s has %zu bytes, %zu needed", what, bytes, need);
  if (((uintptr_t)ws & 255) != 0) return fail(KDA_ERR_WORKSPACE, "%s not 256-byte aligned", what);
  return KDA_OK;
}

// kda_chunk_fwd, with with_ctx kda_chunk_fwd_ctx, and with reuse as well
// kda_chunk_fwd_reuse (the records are already in the context).
kda_status chunk_fwd(const kda_inputs *in, void *o, float *hT, void *ctx, size_t ctx_bytes, bool with_ctx,
                     bool reuse, void *workspace, size_t workspace_bytes, void *stream) {
  g_err[0] = 0;
  Problem P{};
  kda_status st = validate(in, P);
  if (st != KDA_OK) return st;
  const GateArgs ga = gate_args(in);
  if (P.Ttot > 0 && o == nullptr && hT == nullptr)
    return fail(KDA_ERR_INVALID_ARG, "o and hT are NULL (o NULL: the final state alone, which needs hT)");
  if (use_tc(P) && ((uintptr_t)o & 15) != 0)
    return fail(KDA_ERR_INVALID_ARG, "o must be 16-byte aligned (bf16 tensor-core path)");
  const size_t need_ctx = with_ctx ? ctx_layout(P, nullptr, nullptr) : 0;
  with_ctx = need_ctx > 0;
  if ((st = check_ws(need_ctx, ctx, ctx_bytes, "forward context")) != KDA_OK) return st;
  const size_t need = layout(P, ga.on, false, with_ctx, nullptr, nullptr);
  if ((st = check_ws(need, workspace, workspace_bytes)) != KDA_OK) return st;
  if (P.N == 0) return KDA_OK;
  Workspace W;
  layout(P, ga.on, false, with_ctx, (char *)workspace, &W);
  if (with_ctx) ctx_layout(P, (char *)ctx, &W);
  Problem Pg = P;
  cudaError_t e = gate_per_channel(P, ga, W, &Pg, (cudaStream_t)stream);
  if (e == cudaSuccess) {
    if (use_tc(P)) {
      // with o NULL a context call computes the final state alone: the context keeps the records only
      const int mode = o != nullptr ? (kFwdOutput | (with_ctx ? kFwdSave : 0)) : 0;
      e = tc_forward(Pg, ga, W, o, hT, mode, with_ctx && reuse, W.flags + 2, (cudaStream_t)stream);
    } else {
      Problem Pn = Pg;
      e = normalised_copies(Pg, W, &Pn, (cudaStream_t)stream);
      if (e == cudaSuccess) e = simple_forward(Pn, W, o, hT, (cudaStream_t)stream);
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, reuse ? "kda_chunk_fwd_reuse" : with_ctx ? "kda_chunk_fwd_ctx" : "kda_chunk_fwd");
  return KDA_OK;
}

// kda_chunk_bwd, and with with_ctx kda_chunk_bwd_ctx.
kda_status chunk_bwd(const kda_inputs *in, const void *ctx, size_t ctx_bytes, bool with_ctx, const void *dO,
                     const float *dhT, void *dq, void *dk, void *dv, float *dg, float *dbeta, float *dh0,
                     void *workspace, size_t workspace_bytes, void *stream) {
  g_err[0] = 0;
  Problem P{};
  kda_status st = validate(in, P);
  if (st != KDA_OK) return st;
  const GateArgs ga = gate_args(in);
  // dq .. dbeta all NULL with a dh0: the start-state gradient alone (the reverse scan)
  const bool state_only =
      dq == nullptr && dk == nullptr && dv == nullptr && dg == nullptr && dbeta == nullptr && dh0 != nullptr;
  if (P.Ttot > 0 && (dO == nullptr || (!state_only && (dq == nullptr || dk == nullptr || dv == nullptr ||
                                                       dg == nullptr || dbeta == nullptr))))
    return fail(KDA_ERR_INVALID_ARG,
                "dO, dq, dk, dv, dg and dbeta are required (or dq .. dbeta all NULL with dh0: dh0 alone)");
  if (use_tc(P)) {  // the tensor-core kernels load dO by TMA and store the gradients in 4-16 byte vectors
    const char *bad = ((uintptr_t)dO & 15) ? "dO" : ((uintptr_t)dq & 15) ? "dq" : ((uintptr_t)dk & 15) ? "dk"
                      : ((uintptr_t)dv & 15) ? "dv" : (!P.scalar_gate && ((uintptr_t)dg & 15)) ? "dg" : nullptr;
    if (bad != nullptr) return fail(KDA_ERR_INVALID_ARG, "%s must be 16-byte aligned (bf16 tensor-core path)", bad);
  }
  const size_t need_ctx = with_ctx ? ctx_layout(P, nullptr, nullptr) : 0;
  with_ctx = need_ctx > 0;
  if ((st = check_ws(need_ctx, ctx, ctx_bytes, "forward context")) != KDA_OK) return st;
  const size_t need = layout(P, ga.on, true, with_ctx, nullptr, nullptr);
  if ((st = check_ws(need, workspace, workspace_bytes)) != KDA_OK) return st;
  if (P.N == 0) return KDA_OK;
  Workspace W;
  layout(P, ga.on, true, with_ctx, (char *)workspace, &W);
  if (with_ctx) ctx_layout(P, (char *)ctx, &W);  // read only: the context serves any number of backwards
  cudaStream_t s = (cudaStream_t)stream;
  const kda_gate *gate = in->gate;  // (with KDA_GATE_IN_KERNEL; validated)
  Problem Pg = P;
  cudaError_t e = gate_per_channel(P, ga, W, &Pg, s);
  // per-channel gate gradient (a scalar gate's dg is summed over K inside the tensor-core kernel)
  float *dgk = (P.scalar_gate || ga.on) && !use_tc(P) ? W.dgx : dg;
  if (e == cudaSuccess) {
    if (use_tc(P)) {
      int *err = W.flags + 2;
      // the saved tiles come from the context, or from the states pass (the scan alone needs only the records)
      e = with_ctx     ? launch_chunk_map(Pg, W, s)
          : state_only ? tc_records(Pg, ga, W, err, s)
                       : tc_forward(Pg, ga, W, nullptr, nullptr, kFwdSave, false, err, s);
      if (e == cudaSuccess) e = tc_backward_scan(Pg, W, dO, dhT, dh0, err, s);
      if (!state_only) {
        if (e == cudaSuccess) e = tc_backward_intra(Pg, ga, W, dO, dv, dq, dk, dgk, dbeta, err, s);
        if (e == cudaSuccess && P.HV != P.H) e = launch_group_reduce(Pg, W.dqp, W.dkp, dq, dk, s);
        if (e == cudaSuccess && ga.on) e = launch_kgate_param_reduce(Pg, W, gate->dA_log, gate->dbias, s);
      }
    } else {
      Problem Pn = Pg;
      e = normalised_copies(Pg, W, &Pn, s);
      if (e == cudaSuccess) e = simple_backward(Pn, W, dO, dhT, dq, dk, dv, dgk, dbeta, dh0, state_only, s);
    }
  }
  if (e == cudaSuccess && P.scalar_gate && !use_tc(P) && !state_only) e = launch_gate_grad_reduce(P, W.dgx, dg, s);
  if (e == cudaSuccess && ga.on && !use_tc(P) && !state_only)
    e = launch_kgate_grad(P, ga, W, W.dgx, dg, gate->dA_log, gate->dbias, s);
  if (e != cudaSuccess) return cuda_fail(e, with_ctx ? "kda_chunk_bwd_ctx" : "kda_chunk_bwd");
  return KDA_OK;
}

}  // namespace

cudaError_t sm_count(int *out) {
  static std::atomic<int> cached[64];  // zero-initialised; filled once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return cudaSuccess;
}

void set_last_error(const char *msg) {
  strncpy(g_err, msg, sizeof(g_err) - 1);
  g_err[sizeof(g_err) - 1] = 0;
}

}  // namespace kda

using namespace kda;

extern "C" {

size_t kda_chunk_fwd_workspace_size(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return 0;
  return layout(P, gate_args(in).on, false, false, nullptr, nullptr);
}

size_t kda_chunk_bwd_workspace_size(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return 0;
  return layout(P, gate_args(in).on, true, false, nullptr, nullptr);
}

kda_status kda_chunk_fwd(const kda_inputs *in, void *o, float *hT, void *workspace,
                         size_t workspace_bytes, void *stream) {
  return chunk_fwd(in, o, hT, nullptr, 0, false, false, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_bwd(const kda_inputs *in, const void *dO, const float *dhT, void *dq,
                         void *dk, void *dv, float *dg, float *dbeta, float *dh0,
                         void *workspace, size_t workspace_bytes, void *stream) {
  return chunk_bwd(in, nullptr, 0, false, dO, dhT, dq, dk, dv, dg, dbeta, dh0, workspace, workspace_bytes,
                   stream);
}

size_t kda_status_offset(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return ~(size_t)0;
  char *const base = reinterpret_cast<char *>((uintptr_t)1 << 20);  // any aligned address: only offsets are taken
  Workspace W;
  layout(P, gate_args(in).on, false, false, base, &W);
  return (size_t)(reinterpret_cast<char *>(W.flags) - base);  // the same in every workspace layout (it comes first)
}

size_t kda_chunk_ctx_size(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return 0;
  return ctx_layout(P, nullptr, nullptr);
}

size_t kda_chunk_fwd_ctx_workspace_size(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return 0;
  return layout(P, gate_args(in).on, false, ctx_layout(P, nullptr, nullptr) > 0, nullptr, nullptr);
}

size_t kda_chunk_bwd_ctx_workspace_size(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return 0;
  return layout(P, gate_args(in).on, true, ctx_layout(P, nullptr, nullptr) > 0, nullptr, nullptr);
}

kda_status kda_chunk_fwd_ctx(const kda_inputs *in, void *o, float *hT, void *ctx, size_t ctx_bytes,
                             void *workspace, size_t workspace_bytes, void *stream) {
  return chunk_fwd(in, o, hT, ctx, ctx_bytes, true, false, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_fwd_reuse(const kda_inputs *in, void *o, float *hT, void *ctx, size_t ctx_bytes,
                               void *workspace, size_t workspace_bytes, void *stream) {
  return chunk_fwd(in, o, hT, ctx, ctx_bytes, true, true, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_bwd_ctx(const kda_inputs *in, const void *ctx, size_t ctx_bytes, const void *dO,
                             const float *dhT, void *dq, void *dk, void *dv, float *dg, float *dbeta,
                             float *dh0, void *workspace, size_t workspace_bytes, void *stream) {
  return chunk_bwd(in, ctx, ctx_bytes, true, dO, dhT, dq, dk, dv, dg, dbeta, dh0, workspace, workspace_bytes,
                   stream);
}

kda_status kda_recurrent_fwd(const kda_inputs *in, void *o, float *hT, void *stream) {
  g_err[0] = 0;
  Problem P{};
  kda_status st = validate(in, P);
  if (st != KDA_OK) return st;
  if (P.Ttot > 0 && o == nullptr) return fail(KDA_ERR_INVALID_ARG, "o is NULL");
  cudaError_t e = launch_recurrent(P, gate_args(in), o, hT, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_recurrent_fwd");
  return KDA_OK;
}

kda_status kda_state_compose(const float *M, const float *h, const float *c, float *out, int count, int K,
                             int V, int transpose, void *stream) {
  g_err[0] = 0;
  if (count < 0) return fail(KDA_ERR_INVALID_ARG, "count=%d must be >= 0", count);
  if (K < 1 || V < 1) return fail(KDA_ERR_INVALID_ARG, "K=%d V=%d must be positive", K, V);
  if (K > kMaxDim || V > kMaxDim)
    return fail(KDA_ERR_UNSUPPORTED, "K=%d V=%d: dims above %d are not implemented", K, V, kMaxDim);
  if (count == 0) return KDA_OK;
  if (M == nullptr || h == nullptr || out == nullptr) return fail(KDA_ERR_INVALID_ARG, "M, h and out are required");
  const char *o0 = (const char *)out, *o1 = o0 + sizeof(float) * (size_t)count * K * V;
  auto overlaps = [&](const void *p, size_t bytes) {
    const char *a = (const char *)p;
    return a < o1 && o0 < a + bytes;
  };
  if (overlaps(M, sizeof(float) * (size_t)count * K * K) || overlaps(h, sizeof(float) * (size_t)count * K * V))
    return fail(KDA_ERR_INVALID_ARG, "out overlaps M or h");
  cudaError_t e = launch_state_compose(M, h, c, out, count, K, V, transpose != 0, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_state_compose");
  return KDA_OK;
}

const char *kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported problem";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char *kda_last_error(void) { return g_err; }

int kda_version(void) { return 107; }

int kda_uses_tensor_cores(const kda_inputs *in) {
  Problem P{};
  if (validate(in, P) != KDA_OK) return -1;
  return use_tc(P) ? 1 : 0;
}

}  // extern "C"
