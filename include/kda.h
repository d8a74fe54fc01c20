/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked KDA library (libkda.so).
 *
 * KDA (Kimi Delta Attention) is a gated delta-rule recurrence with a
 * per-channel decay.  For every logical sequence n and value head j an fp32
 * state S[K][V] evolves token by token:
 *     S <- diag(2^g_t) S                       (g_t: per-token, per-channel log2 decay)
 *     S <- S + beta_t k_t (v_t - S^T k_t)^T    (delta-rule write, prediction from the decayed state)
 *     o_t = S^T (q_t / sqrt(K))                (read-out from the updated state)
 * The chunked entry points evaluate this exactly (up to rounding) in chunks of
 * 64 tokens: a chunk-local gate cumsum, the strictly-lower decayed beta*K*K^T
 * block L and its unit-lower inverse A = (I+L)^-1, w = A(beta k 2^G),
 * u = A(beta v), an inter-chunk state scan and the output o = (q 2^G) h + Aqk(u - w h).
 * This is the sub-kernel decomposition of the FLA KDA/GDN pipeline
 * (chunk_scaled_dot_kkt / solve_tril / recompute_w_u / fwd_h / fwd_o, and
 * bwd_dhu / bwd_dqkwg / bwd_dv_local / wy_bwd for the backward) named in
 * "[Fix] Use unit KDA gate scale when A_log is omitted"
 * (fla-org/flash-linear-attention PR #1294, commit log, GDN per-kernel tests).
 *
 * Argument contract (mirrors the recurrent_kda / chunk_kda contract in
 * "kda in torchtitan (training)", pytorch/torchtitan PR #4164, agent note):
 *   - the gate g is the PER-TOKEN log2 decay (the library does the chunk cumsum);
 *   - queries are scaled by 1/sqrt(K) internally;
 *   - cu_seqlens is a DEVICE int32 array of N+1 non-decreasing offsets with
 *     cu_seqlens[0] == 0 and cu_seqlens[N] <= T; repeated offsets are empty
 *     slots whose state passes through bitwise (hT[n] = h0[n], dh0[n] = dhT[n]);
 *     tokens at or after cu_seqlens[N] are outside the contract: never read for
 *     a result and never written;
 *   - states are fp32 with one leading entry per logical sequence.
 *
 * Layouts (row-major, all DEVICE pointers):
 *   q, k, dq, dk   [B][T][H][K]      dtype
 *   v, o, dO, dv   [B][T][HV][V]     dtype
 *   g, dg          [B][T][HV][K]     fp32  ([B][T][HV] with KDA_SCALAR_GATE)
 *   beta, dbeta    [B][T][HV]        fp32
 *   h0,hT,dhT,dh0  [N][HV][K][V]     fp32
 * bf16 problems with K and V each 64 or 128 run the tensor-core kernels when
 * q, k, v and g are 16-byte aligned (they arrive by TMA; a 64-wide head runs
 * zero-padded in the 128-wide tiles); otherwise the general kernels run, with
 * the same results (kda_uses_tensor_cores() tells which).  On the tensor-core
 * path o, dO, dq, dk, dv and (per-channel gate) dg must be 16-byte aligned too
 * (KDA_ERR_INVALID_ARG otherwise).
 * Value head j reads query/key head j / (HV/H) (contiguous groups).
 * dq and dk are summed over the HV/H value heads that share a q/k head.
 *
 * Ownership: the caller allocates every input, output and workspace buffer;
 * the library never allocates or frees device memory, never synchronises and
 * never reads device data on the host.  Work is enqueued on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).  kda_chunk_bwd
 * recomputes everything it needs from the inputs; the _ctx pair instead keeps
 * the forward's intermediates in a caller-owned context buffer.
 *
 * Errors: arguments the host can check are validated before anything is
 * enqueued and reported synchronously (KDA_ERR_INVALID_ARG,
 * KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE); nothing is launched in that case.
 * A failed launch returns KDA_ERR_CUDA.  kda_last_error() returns a message
 * for the last failure on the calling thread.  The values inside cu_seqlens
 * live on the device and are a precondition: they are not checked.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null required pointer, bad sizes, HV % H != 0, ... */
  KDA_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement     */
  KDA_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than required  */
  KDA_ERR_CUDA = 4         /* a CUDA launch or API call failed                 */
} kda_status;

typedef enum kda_dtype {
  KDA_F32 = 0,  /* q, k, v (and o, dO, dq, dk, dv) in fp32: fp32 arithmetic throughout */
  KDA_BF16 = 1  /* q, k, v (and o, dO, dq, dk, dv) in bf16: fp32 accumulation          */
} kda_dtype;

/* Bits of kda_inputs.flags. */
enum {
  /* q/k L2-norm prologue: each (token, q/k head) row of q and of k is divided
   * by sqrt(sum over the K channels of its squares + 1e-6) before the op (and
   * before the 1/sqrt(K) query scale); dq and dk are then gradients w.r.t. the
   * raw rows.  The KDA layer of "kda in torchtitan (training)"
   * (pytorch/torchtitan PR #4164) imports such an `l2norm` beside
   * `recurrent_kda`; its epsilon is not printed there (1e-6 is this library's
   * choice). */
  KDA_QK_L2NORM = 1,
  /* scalar gate (the GDN variant): g and dg are [B][T][HV] fp32, one log2 decay
   * per (token, value head) shared by every key channel -- the gated delta rule
   * of the GDN pipeline named in "[Fix] Use unit KDA gate scale when A_log is
   * omitted" (fla-org/flash-linear-attention PR #1294, commit log), of which
   * KDA's per-channel gate is the generalisation.  dg is the sum over K of the
   * per-channel gradients. */
  KDA_SCALAR_GATE = 2,
  /* KDA gate inside the op: `g` holds the raw gate pre-activations a (same
   * layout, fp32) and `gate` the gate's parameters; the op makes the per-token
   * log2 decay itself, with x = a + bias and s = exp(A_log):
   *   unbounded (lower_bound == 0):  g = -s softplus(x)
   *   bounded   (lower_bound  < 0):  g = lower_bound sigmoid(s x)
   * An omitted A_log is a unit scale, the same as an explicit zero A_log
   * ("[Fix] Use unit KDA gate scale when A_log is omitted",
   * fla-org/flash-linear-attention PR #1294, Summary and Breaking changes; the
   * page prints no formula: the two above are this library's reading).  The
   * backward's dg is then the gradient w.r.t. a, and the gate's parameter
   * gradients are summed over every valid token in fp32 (that page's commit
   * log: gate bias gradients reduced in fp32 before any downcast).  Not
   * combined with KDA_SCALAR_GATE (KDA_ERR_UNSUPPORTED). */
  KDA_GATE_IN_KERNEL = 4
};

/* Parameters of the KDA gate (KDA_GATE_IN_KERNEL); DEVICE pointers. */
typedef struct kda_gate {
  const float *A_log; /* [HV] log of the decay scale, or NULL: unit scale (the same as zeros) */
  const float *bias;  /* [HV][K] added to a, or NULL                                       */
  float lower_bound;  /* 0: the unbounded gate; < 0: the bounded gate (finite)              */
  float *dA_log;      /* backward output [HV] (fp32), or NULL                                */
  float *dbias;       /* backward output [HV][K] (fp32), or NULL                             */
} kda_gate;

/* Problem description shared by every entry point.  Zero-initialise it: a
 * zero flags field keeps the plain behaviour. */
typedef struct kda_inputs {
  int B, T;         /* batch and (padded) tokens per batch row; B must be 1 with cu_seqlens */
  int H, HV;        /* query/key heads and value heads; HV must be a multiple of H          */
  int K, V;         /* key and value head dims: 1..128 each (tensor cores: 64 or 128, bf16)   */
  int N;            /* logical sequences: B when cu_seqlens is NULL, else len(cu_seqlens)-1   */
  kda_dtype dtype;  /* element type of q, k, v, o, dO, dq, dk, dv                            */
  const void *q, *k, *v;
  const float *g;           /* per-token log2 decay: any finite value <= 0                    */
  const float *beta;        /* per (token, value head) write strength                        */
  const float *h0;          /* initial states [N][HV][K][V], or NULL for zeros               */
  const int32_t *cu_seqlens;/* device [N+1] packed offsets, or NULL for a dense batch         */
  int flags;                /* KDA_QK_L2NORM | KDA_SCALAR_GATE | KDA_GATE_IN_KERNEL, or 0;   */
                            /* other bits: KDA_ERR_INVALID_ARG                                 */
  const kda_gate *gate;     /* host pointer; required with KDA_GATE_IN_KERNEL, else ignored   */
} kda_inputs;

/* Bytes of device workspace kda_chunk_fwd needs for this problem (256-byte
 * aligned base required).  Returns 0 if the problem is invalid. */
size_t kda_chunk_fwd_workspace_size(const kda_inputs *in);

/* Chunked forward.  Writes o [B][T][HV][V] (dtype) for every valid token and,
 * if hT is not NULL, the final states hT [N][HV][K][V] (fp32).  o may be NULL
 * when hT is not: then only the final states are computed (no output work).
 * workspace: device scratch of at least kda_chunk_fwd_workspace_size() bytes;
 * its contents on entry do not matter and are clobbered. */
kda_status kda_chunk_fwd(const kda_inputs *in, void *o, float *hT, void *workspace,
                         size_t workspace_bytes, void *stream);

/* Bytes of device workspace kda_chunk_bwd needs. */
size_t kda_chunk_bwd_workspace_size(const kda_inputs *in);

/* Chunked backward with state recompute.  Given dO [B][T][HV][V] (dtype) and the
 * final-state gradient dhT [N][HV][K][V] (fp32, NULL = zero), writes
 * dq, dk [B][T][H][K] (dtype), dv [B][T][HV][V] (dtype), dg [B][T][HV][K] (fp32,
 * gradient w.r.t. the log2 gate), dbeta [B][T][HV] (fp32) for every valid token
 * and, if dh0 is not NULL, dh0 [N][HV][K][V] (fp32).  With dq, dk, dv, dg and
 * dbeta all NULL and dh0 not NULL, only dh0 is computed (the initial-state
 * gradient alone: the reverse state scan, none of the per-token gradient
 * work) -- what a context-parallel rank needs before its relay. */
kda_status kda_chunk_bwd(const kda_inputs *in, const void *dO, const float *dhT, void *dq,
                         void *dk, void *dv, float *dg, float *dbeta, float *dh0,
                         void *workspace, size_t workspace_bytes, void *stream);

/* ---- forward context: the backward without its recompute (no counterpart on
 * the pages, which leave open what a forward keeps for its backward) ----
 * On the tensor-core path (bf16, K, V = 64 or 128, aligned q/k/v/g) the backward
 * first re-runs two forward kernels: the per-chunk record kernel and the
 * state chain that saves every chunk's start state.  kda_chunk_fwd_ctx writes
 * those results into a caller-owned context buffer while it computes o, and
 * kda_chunk_bwd_ctx reads them from it instead: same results, bit for bit, as
 * kda_chunk_fwd + kda_chunk_bwd, for kda_chunk_ctx_size() bytes of device
 * memory per layer -- per (64-token chunk, value head): the 66,048-byte record
 * (decayed key and query tiles, the inverse A, Aqk, 2^G_last), the bf16
 * chunk-start state (32 KB) and two 16 KB bf16 tiles (X^T, D^T).  A _ctx or
 * _reuse forward with o NULL computes the final states alone: it leaves the
 * context holding the records only, and a backward needs a later forward on
 * the context with o.
 * The context must come from kda_chunk_fwd_ctx on the same inputs (q, k, v,
 * g, beta, h0, cu_seqlens, flags), unchanged since; that is a precondition,
 * not checked.  The backward only reads it, so it serves any number of
 * backward calls.  Both calls require a 256-byte aligned context of at least
 * kda_chunk_ctx_size() bytes (KDA_ERR_WORKSPACE otherwise).  On the general
 * path kda_chunk_ctx_size() is 0, nothing is kept, ctx may be NULL and the
 * _ctx calls behave as kda_chunk_fwd / kda_chunk_bwd. */

/* Bytes of forward context for this problem (0: general path, or invalid). */
size_t kda_chunk_ctx_size(const kda_inputs *in);

/* Workspace of kda_chunk_fwd_ctx / kda_chunk_bwd_ctx: the plain sizes minus
 * the regions the context holds. */
size_t kda_chunk_fwd_ctx_workspace_size(const kda_inputs *in);
size_t kda_chunk_bwd_ctx_workspace_size(const kda_inputs *in);

/* kda_chunk_fwd that also fills ctx. */
kda_status kda_chunk_fwd_ctx(const kda_inputs *in, void *o, float *hT, void *ctx, size_t ctx_bytes,
                             void *workspace, size_t workspace_bytes, void *stream);

/* kda_chunk_fwd_ctx for inputs that share q, k, g, beta, cu_seqlens, flags and
 * sizes with the ones ctx was last filled from (v and h0 may differ): the
 * per-chunk records, which depend on those alone, are read from ctx instead of
 * recomputed -- the several passes of a context-parallel rank over one segment.
 * With o not NULL the chunk-start states and tiles in ctx are rewritten for
 * these inputs, so the context then serves their backward.  On the general
 * path: kda_chunk_fwd. */
kda_status kda_chunk_fwd_reuse(const kda_inputs *in, void *o, float *hT, void *ctx, size_t ctx_bytes,
                               void *workspace, size_t workspace_bytes, void *stream);

/* kda_chunk_bwd on the context kda_chunk_fwd_ctx filled (read only). */
kda_status kda_chunk_bwd_ctx(const kda_inputs *in, const void *ctx, size_t ctx_bytes, const void *dO,
                             const float *dhT, void *dq, void *dk, void *dv, float *dg, float *dbeta,
                             float *dh0, void *workspace, size_t workspace_bytes, void *stream);

/* Token-by-token recurrent forward (inference): one sequential pass per
 * (sequence, value head), fp32 state and fp32 arithmetic whatever the dtype,
 * no workspace.  Same arguments and results as kda_chunk_fwd, as in the
 * recurrent_kda entry point of "kda in torchtitan (training)". */
kda_status kda_recurrent_fwd(const kda_inputs *in, void *o, float *hT, void *stream);

/* State composition for the context-parallel state relay.  When a sequence is
 * split across ranks, each rank's segment maps the state it starts from
 * affinely, S_end = M S_start + c: c is the segment's final state from a zero
 * start and M (K x K) the segment's transition, which kda_chunk_fwd returns
 * as hT when run on the segment with v = 0, V = K and h0 = the identity.  An
 * exclusive scan of out = M h + c across ranks gives every rank its true start
 * state, and the backward scan uses out = M^T dh + c on state gradients: the
 * synchronous context parallelism of "[KDA] Add Paddle training compatibility"
 * (PFCCLab/flash-linear-attention PR #2, summary and test plan).
 *   M    [count][K][K] fp32     h, out [count][K][V] fp32     c [count][K][V] fp32 or NULL (zero)
 *   out[i] = op(M[i]) h[i] + c[i], op = transpose when `transpose` != 0.
 * DEVICE pointers; out may equal c but must not overlap M or h.  count >= 0,
 * 1 <= K, V <= 128; violations are KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED
 * before anything is launched. */
kda_status kda_state_compose(const float *M, const float *h, const float *c, float *out, int count, int K,
                             int V, int transpose, void *stream);

/* Device status words of a call.  Every chunked call (forward, backward, any
 * variant) writes seven int32 words into its workspace, at byte offset
 * kda_status_offset() (the same for every workspace of the problem):
 *   [0] the number of 64-token chunks mapped;
 *   [1] nonzero if cu_seqlens was malformed (decreasing, negative or past the
 *       token axis): those sequences were treated as empty;
 *   [2] nonzero if a bounded device wait gave up (a copy or product never
 *       completed): the call's results are invalid;
 *   [3] the (chunk, value head) slots whose forward records took the exact
 *       path for strong decays, and
 *   [4] those whose per-chunk gradients took it;
 *   [5] the slots whose per-chunk gradients took the 16-token block path, and
 *   [6] those whose forward records took it (tensor-core path only for 3..6).
 *       The kernels split each pairwise decay 2^(G_r - G_i) of a chunk at one
 *       reference per channel, the middle of the channel's range over the
 *       chunk; a chunk whose decay span (the sum of 63 consecutive per-token
 *       gates of one channel) exceeds 192 (log2) is recomputed by a second
 *       launch with references inside its 16-token blocks, and a block whose
 *       span (15 gates) exceeds 192 by a third, slower launch that forms the
 *       block's terms exactly.  Results are exact for any gate either way;
 *       the words only say where time went.
 * Words 2 to 6 are cleared at the start of every call.  The library never
 * reads them on the host: copy them out after the call (in stream order) to
 * check.  Returns SIZE_MAX for an invalid problem. */
size_t kda_status_offset(const kda_inputs *in);

/* Which kernels a call on these inputs runs: 1 for the tensor-core kernels
 * (bf16, K and V each 64 or 128, with q, k, v and a per-channel g 16-byte
 * aligned), 0 for the general fp32 kernels (same results, several times
 * slower), -1 if the problem is invalid.  A bf16 problem whose inputs are a
 * slice of a larger tensor starting off a 16-byte boundary runs the general
 * kernels: this tells the caller so before the call. */
int kda_uses_tensor_cores(const kda_inputs *in);

/* Static description of a status code. */
const char *kda_status_string(kda_status s);

/* Message describing the last failure on the calling thread ("" if none). */
const char *kda_last_error(void);

/* Library ABI version (major * 100 + minor): 107 (101: kda_inputs gained
 * `flags`; 102: the forward-context entry points; 103: the final-state-only
 * forward, the start-state-gradient-only backward, kda_chunk_fwd_reuse; 104:
 * kda_status_offset, kda_debug_bounded_wait; 105: status words 3 and 4,
 * kda_uses_tensor_cores; 106: KDA_GATE_IN_KERNEL and kda_inputs.gate; 107:
 * status words 5 and 6). */
int kda_version(void);

/* Chunked forward without a caller workspace (no counterpart on the pages).
 * For callers that cannot allocate device memory -- a host program linked
 * against this library alone, a runtime that plans every device byte at
 * start-up and forbids allocation afterwards -- this runs kda_chunk_fwd on a
 * scratch array that lives inside the library: 4 MiB of device memory per GPU
 * that loads it, held until the process exits.  Same arguments and results as
 * kda_chunk_fwd minus the workspace.  The first call on a device looks up the
 * array's address with that device current and keeps it for the life of the
 * process; make it before any CUDA-graph capture, and do not reset the device
 * (cudaDeviceReset) after it.  All calls share the one array (it keeps the
 * last call's contents; nothing in it must start at zero), so calls that may
 * overlap on the GPU race: order them on one stream.  A problem whose workspace exceeds 4 MiB is
 * rejected with KDA_ERR_WORKSPACE before anything is launched.  The library
 * allocates nothing on this path. */
kda_status kda_chunk_fwd_noalloc(const kda_inputs *in, void *o, float *hT, void *stream);

/* ---- instrumentation (benchmarks and profiling; no counterpart on the pages) ----
 * Every kernel the library launches is counted.  While timing is enabled, a
 * CUDA event pair is recorded on the launching stream around each launch. */

/* Runs one device thread that waits, bounded by `polls` polls (1 .. 2^24), on
 * an mbarrier that nothing completes: the wait gives up and sets *err (a device
 * int) to 1, the way a kernel of this library reports a copy that never
 * arrived.  For tests of that path; it neither faults nor hangs the GPU. */
kda_status kda_debug_bounded_wait(int *err, long long polls, void *stream);

/* Kernels launched by this library in this process so far. */
unsigned long long kda_launch_count(void);

/* Turns per-launch event timing on (1) or off (0); returns the previous state. */
int kda_timing_enable(int on);

/* Waits for every recorded event pair, sums the elapsed times per kernel name and
 * clears the records.  Fills up to max_kernels entries: names (each name_stride
 * bytes, NUL-terminated), total milliseconds and launch counts.  Returns the
 * number of distinct kernels seen (may exceed max_kernels). */
int kda_timing_collect(int max_kernels, char *names, size_t name_stride, double *total_ms,
                       int *launches);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
