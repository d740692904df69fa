/*
 * lowrank.h — C ABI of liblowrank.so, the GB300 (sm_103a) implementation of the
 * low-rank bottleneck sublayer trained by BOOST.
 *
 * Source of the method: "BOOST: BOttleneck-Optimized Scalable Training Framework
 * for Low-Rank Large Language Models" (arXiv 2512.12131; abstract, and the
 * gist.science technical summary §1-§2).  Every dense linear map W.x of the model
 * is replaced by a low-rank pair — an r x d_in layer A followed by a d_out x r
 * layer B (technical summary §1, §2.1) — which this library evaluates as
 *
 *     y = B . SiLU(A . v)                                  (one "pair")
 *
 * and the three system optimisations of technical summary §2.2 are built in:
 *   - Online-RMSNorm: the RMSNorm gain is folded into A, the sum of squares of
 *     the input row is accumulated alongside the first GEMM and the 1/rms row
 *     scale is applied in that GEMM's epilogue (exact rewrite of RMSNorm);
 *   - linear-layer grouping: A's that read the same input (gate/up, q/k/v)
 *     are concatenated into one GEMM; the B's with distinct inputs run as one
 *     batched GEMM;
 *   - low-rank activation checkpointing: in LR_SAVE_CKPT mode only the block
 *     input, the [T, r] bottleneck pre-activations and 1/rms are kept; the
 *     backward recomputes the rest inside the block.
 *
 * Conventions for every entry point
 *   - Matrices are dense row-major; a token is one row.  x is [T, d].  A pair's
 *     A is [r, d_in] and its B is [d_out, r].  No biases.
 *   - lr_dtype selects the storage and arithmetic: LR_BF16 stores every tensor
 *     in bf16 and runs tcgen05 tensor-core GEMMs with fp32 accumulation;
 *     LR_F32 stores fp32 and runs exact fp32 (SIMT) GEMMs.  Weight gradients and
 *     dg are always fp32.  1/rms (s) is always fp32.
 *   - All pointers are DEVICE pointers of the current CUDA device, 16-byte
 *     aligned.  d, d_in, d_out, f and r must be positive multiples of 8; T >= 1.
 *   - Ownership: the caller allocates and owns every buffer, including `saved`
 *     and the workspace `ws` (sizes from the *_bytes queries, which need no
 *     device).  The library allocates and frees nothing and never synchronises,
 *     except lr_check_device_error.  Outputs must not alias inputs.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); all work is
 *     enqueued on it, asynchronously.  The checkpointed bf16 MLP backward also
 *     runs two of its kernels on a second stream of the library's (one per host
 *     thread and device, created on the first such call and kept), forked from
 *     `stream` and joined back to it with events inside the call: to the caller
 *     all work stays ordered on `stream`, and graph capture of `stream` takes it
 *     in.
 *   - Errors: arguments are validated before any launch; on failure the call
 *     returns a non-zero lr_status, launches nothing and leaves a message in
 *     lr_last_error() (thread-local).  A failed launch returns LR_ERR_CUDA.
 *     Kernels never trap: a bounded wait that runs out sets a device error
 *     word, which lr_check_device_error reports as LR_ERR_TIMEOUT.
 *   - Results are deterministic: the same inputs give the same bits (no atomics
 *     in any reduction; the attention kernels take work items from an atomic
 *     counter, but an item's result does not depend on who computes it), so LR_SAVE_CKPT and LR_SAVE_FULL give bitwise-equal
 *     gradients.
 */
#ifndef LOWRANK_H_
#define LOWRANK_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LR_OK = 0,
  LR_ERR_NULL = 1,        /* a required pointer is NULL */
  LR_ERR_SHAPE = 2,       /* a dimension is non-positive, not a multiple of 8, or too large */
  LR_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  LR_ERR_DTYPE = 4,       /* unknown lr_dtype, lr_mode or lr_act */
  LR_ERR_WORKSPACE = 5,   /* saved / ws buffer smaller than the size query returns */
  LR_ERR_CUDA = 6,        /* a CUDA call or kernel launch failed */
  LR_ERR_TIMEOUT = 7,     /* a kernel's bounded wait ran out (reported by lr_check_device_error) */
  LR_ERR_UNSUPPORTED = 8  /* no usable device / architecture */
} lr_status;

typedef enum { LR_F32 = 0, LR_BF16 = 1 } lr_dtype;

typedef enum {
  LR_SAVE_FULL = 0, /* keep every forward intermediate for the backward */
  LR_SAVE_CKPT = 1  /* low-rank activation checkpointing (technical summary §2.2) */
} lr_mode;

/* The activation sigma between a pair's A and B.  The pages name no sigma: SiLU is the
 * reading used throughout; identity is the plain factorisation W = B A (the SVD-style
 * low-rank variant the technical summary lists).  The SwiGLU product of the MLP block
 * keeps its SiLU in both. */
typedef enum { LR_ACT_SILU = 0, LR_ACT_IDENTITY = 1 } lr_act;

/* One low-rank pair: A [r, d_in] and B [d_out, r], storage dtype. */
typedef struct {
  const void* A;
  const void* B;
} lr_pair;

/* Gradients of one pair, fp32, same shapes as the weights. */
typedef struct {
  float* dA;
  float* dB;
} lr_pair_grad;

/* ------------------------------------------------------------------ MLP block
 * Low-rank SwiGLU MLP block with a residual (the sublayer the technical summary
 * §2.2 groups as gate/up down-projections plus a down pair):
 *     n   = RMSNorm(x; g, eps)              s[t] = (mean_j x[t,j]^2 + eps)^(-1/2)
 *     a   = B_gate sigma(A_gate n)          A_gate [r,d],  B_gate [f,r]
 *     b   = B_up   sigma(A_up   n)          A_up   [r,d],  B_up   [f,r]
 *     h   = SiLU(a) * b                     [T, f]
 *     out = x + B_down sigma(A_down h)      A_down [r,f],  B_down [d,r]
 * Dimensions: T tokens, d model width, f MLP width, r rank; sigma per `act`.
 *
 * `saved` holds what the backward needs: in LR_SAVE_CKPT the pre-activations
 * u_gate, u_up, u_down ([T, r] each, dtype) and s ([T] fp32); LR_SAVE_FULL adds
 * the sigma outputs and a, b, h.  Its layout is private; pass it unchanged to
 * lr_mlp_bwd with the same dtype, mode, act and dimensions.  x must also be passed
 * unchanged to the backward (checkpointing keeps the block input, not a copy).
 */
size_t lr_mlp_saved_bytes(lr_dtype dt, lr_mode mode, int T, int d, int f, int r);
size_t lr_mlp_fwd_workspace_bytes(lr_dtype dt, lr_mode mode, int T, int d, int f, int r);
size_t lr_mlp_bwd_workspace_bytes(lr_dtype dt, lr_mode mode, int T, int d, int f, int r);

/* x [T,d], g [d] -> out [T,d]; fills `saved`. */
lr_status lr_mlp_fwd(lr_dtype dt, lr_mode mode, lr_act act, int T, int d, int f, int r, float eps, const void* x,
                     const void* g, lr_pair gate, lr_pair up, lr_pair down, void* out, void* saved,
                     size_t saved_bytes, void* ws, size_t ws_bytes, void* stream);

/* dout [T,d] = dL/dout -> dx [T,d] (dtype), dg [d] fp32, and every pair's dA, dB (fp32).
 * In LR_SAVE_CKPT the backward first re-runs the block's forward from x, s and
 * the saved pre-activations (no other state). */
lr_status lr_mlp_bwd(lr_dtype dt, lr_mode mode, lr_act act, int T, int d, int f, int r, float eps, const void* x,
                     const void* g, lr_pair gate, lr_pair up, lr_pair down, const void* saved,
                     size_t saved_bytes, const void* dout, void* dx, float* dg, lr_pair_grad dgate,
                     lr_pair_grad dup, lr_pair_grad ddown, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- projection group
 * `group` (1..3) pairs that read the same input x [T, d_in], each mapping to
 * d_out (attention q/k/v; technical summary §2.2 grouping):
 *     v = RMSNorm(x; g, eps) if g != NULL, else v = x
 *     outs[i] = B_i sigma(A_i v)           A_i [r, d_in], B_i [d_out, r]; sigma per `act`
 * The A_i run as one stacked GEMM, the B_i as one batched GEMM.  `saved` keeps
 * the stacked pre-activations [T, group*r], the sigma outputs and s.
 */
size_t lr_proj_saved_bytes(lr_dtype dt, int T, int d_in, int d_out, int r, int group, int norm);
size_t lr_proj_fwd_workspace_bytes(lr_dtype dt, int T, int d_in, int d_out, int r, int group, int norm);
size_t lr_proj_bwd_workspace_bytes(lr_dtype dt, int T, int d_in, int d_out, int r, int group, int norm);

lr_status lr_proj_fwd(lr_dtype dt, lr_act act, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                      const void* g, float eps, const void* x, void* const* outs, void* saved, size_t saved_bytes,
                      void* ws, size_t ws_bytes, void* stream);

/* douts[i] [T, d_out] -> dx [T, d_in] (dtype), dg [d_in] fp32 (ignored and may be NULL
 * when g == NULL), grads[i] (fp32). */
lr_status lr_proj_bwd(lr_dtype dt, lr_act act, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                      const void* g, float eps, const void* x, const void* saved, size_t saved_bytes,
                      const void* const* douts, void* dx, float* dg, const lr_pair_grad* grads, void* ws,
                      size_t ws_bytes, void* stream);

/* ------------------------------------------------------- dense MLP block
 * The full-rank block that the low-rank MLP block replaces (the pages compare
 * BOOST against full-rank training; this is the same-device reference point):
 *     n   = RMSNorm(x; g, eps)
 *     a   = W_gate n,  b = W_up n           W_gate, W_up [f, d]
 *     h   = SiLU(a) * b                     [T, f]
 *     out = x + W_down h                    W_down [d, f]
 * It runs on the same kernels as the low-rank block: gate/up as one
 * dual-accumulator GEMM with the gain folded into the weights and 1/rms applied
 * as a row scale (s from a row pass), the SwiGLU product and its backward fused
 * into the GEMM epilogues.  `saved` keeps a, b, h (dtype) and s (fp32); there
 * is no checkpointing mode.  Same conventions and errors as the MLP block.
 */
size_t lr_dense_saved_bytes(lr_dtype dt, int T, int d, int f);
size_t lr_dense_fwd_workspace_bytes(lr_dtype dt, int T, int d, int f);
size_t lr_dense_bwd_workspace_bytes(lr_dtype dt, int T, int d, int f);

/* x [T,d], g [d] -> out [T,d]; fills `saved`. */
lr_status lr_dense_fwd(lr_dtype dt, int T, int d, int f, float eps, const void* x, const void* g,
                       const void* W_gate, const void* W_up, const void* W_down, void* out, void* saved,
                       size_t saved_bytes, void* ws, size_t ws_bytes, void* stream);

/* dout [T,d] -> dx [T,d] (dtype), dg [d], dW_gate, dW_up [f,d], dW_down [d,f] (fp32). */
lr_status lr_dense_bwd(lr_dtype dt, int T, int d, int f, float eps, const void* x, const void* g,
                       const void* W_gate, const void* W_up, const void* W_down, const void* saved,
                       size_t saved_bytes, const void* dout, void* dx, float* dg, float* dW_gate, float* dW_up,
                       float* dW_down, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------- bottleneck-aware tensor parallelism (BTP)
 * BTP (technical summary §2.1) keeps activations sharded along d across the
 * tensor-parallel ranks and runs a normed group of A's row-parallel: each rank
 * reduces over its own d-shard, and the one collective is an all-reduce at the
 * bottleneck width r instead of d.  Online-RMSNorm (§2.2) defers the
 * normalisation and carries the RMS statistics on that same all-reduce.  These
 * two calls are one rank's compute around that all-reduce (which the caller
 * runs, e.g. NCCL over `payload`):
 *
 * lr_btp_partial: x_shard [T, d_shard], g_shard [d_shard] and the d_shard
 *   columns of each pairs[i].A ([r, d_shard], row-major; pairs[i].B unused)
 *   -> payload, fp32, lr_btp_payload_floats(T, r, group) floats:
 *      acc [T, group*r] = x_shard (A_shard * g_shard)^T   (partial sums), then
 *      ss  [T]          = sum_j x_shard[t, j]^2           (partial statistics).
 * lr_btp_finish: the payload summed over all ranks, d = the full width ->
 *      s = (ss / d + eps)^(-1/2), u = round(s acc), z = sigma(u)  ([T, group*r]
 *   dtype, s [T] fp32): what lr_proj_fwd's normed group computes unsharded.
 * ws of lr_btp_partial: lr_btp_workspace_bytes (the folded A shard).
 */
size_t lr_btp_payload_floats(int T, int r, int group);
size_t lr_btp_workspace_bytes(lr_dtype dt, int d_shard, int r, int group);
lr_status lr_btp_partial(lr_dtype dt, int T, int d_shard, int r, int group, const lr_pair* pairs,
                         const void* g_shard, const void* x_shard, float* payload, void* ws, size_t ws_bytes,
                         void* stream);
lr_status lr_btp_finish(lr_dtype dt, lr_act act, int T, int d, int r, int group, const float* payload, float eps,
                        void* u, void* z, float* s, void* stream);

/* ------------------------------------------------ causal self-attention
 * The technical summary trains low-rank LLaMA-style transformers: between the q/k/v
 * projection group and the o-projection sits ordinary causal softmax attention, which
 * the method leaves unchanged.  Per batch entry and head (b entries of s tokens, H heads
 * of dh channels):
 *     S = scale Q K^T (S_ij = -inf for j > i),  P = softmax_j(S),  O = P V,
 * and the backward of sum(O * dO):
 *     dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 * q, k, v, o, dout, dq, dk, dv: [b*s, H*dh] bf16, token-major as the projections write
 * them (head h of token t in columns h*dh .. h*dh + dh - 1 of row t = batch*s + position).
 * saved: lr_attn_saved_bytes (the row log-sum-exp of S, fp32 [b*H*s]); the backward
 * recomputes S from q and k.  ws: lr_attn_workspace_bytes, owned by the caller: for dh = 128
 * (the kernels that keep the scores on chip) a work-item counter, scale dS^T in bf16
 * [b*H*s keys, s queries] (written by the backward for its dQ GEMM) and D in fp32 [b*H*s]:
 * 2 b*H*s*s + 4 b*H*s bytes plus alignment; for other dh the head-major scores [b*H*s, s]
 * (S in fp32, whose first half holds dS in bf16 during the backward, P in bf16) and D:
 * 6 b*H*s*s + 4 b*H*s bytes plus alignment.  The
 * kernels read q, k, v, o, dout and write o, dq, dk, dv in place.  bf16 only (LR_F32:
 * LR_ERR_UNSUPPORTED).  s a multiple of 256, dh a multiple of 128, b*H*s at most 2^30 and
 * b*H*s*s at most 2^40 (LR_ERR_SHAPE otherwise); pointers 16-byte aligned (LR_ERR_ALIGN).
 */
size_t lr_attn_saved_bytes(int b, int s, int H, int dh);
size_t lr_attn_workspace_bytes(int b, int s, int H, int dh);
lr_status lr_attn_fwd(lr_dtype dt, int b, int s, int H, int dh, float scale, const void* q, const void* k,
                      const void* v, void* o, void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                      void* stream);
lr_status lr_attn_bwd(lr_dtype dt, int b, int s, int H, int dh, float scale, const void* q, const void* k,
                      const void* v, const void* o, const void* saved, const void* dout, void* dq, void* dk,
                      void* dv, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------- low-rank transformer block
 * One pre-norm LLaMA-style block whose linear maps are all low-rank pairs (d = H*dh,
 * T = b*s tokens, attention rank ra, MLP rank rm, MLP width f):
 *     [q; k; v] = LR_{q,k,v}(RMSNorm(x; g_attn))       (one normed group, as lr_proj_fwd)
 *     o = causal attention(q, k, v), scale 1/sqrt(dh)  (as lr_attn_fwd)
 *     x1 = x + LR_o(o)                                 (LR = B SiLU(A .), no norm)
 *     out = MLP block(x1; g_mlp, gate, up, down)       (as lr_mlp_fwd, LR_SAVE_CKPT)
 * lr_block_bwd returns dx and every gradient (fp32; the gains' dg_attn, dg_mlp [d]).
 * x, out, dout, dx: [T, d] bf16; all pairs' shapes follow lr_pair (q, k, v, o: A [ra, d],
 * B [d, ra]; gate, up: A [rm, d], B [f, rm]; down: A [rm, f], B [d, rm]).  saved keeps the
 * pieces' saved sets plus q, k, v, o and x1 ([T, d] each); ws is shared by the pieces.
 * bf16 only; the shape rules of lr_attn_fwd and lr_mlp_fwd apply.  lr_attn_* and lr_block_* launch
 * their kernels without programmatic dependent launch (each kernel starts after the previous
 * one completes): with it, three block steps issued back to back stopped making progress.
 */
typedef struct {
  const void* g_attn;
  lr_pair q, k, v, o;
  const void* g_mlp;
  lr_pair gate, up, down;
} lr_block_weights;

typedef struct {
  float* dg_attn;
  lr_pair_grad q, k, v, o;
  float* dg_mlp;
  lr_pair_grad gate, up, down;
} lr_block_grads;

size_t lr_block_saved_bytes(int b, int s, int H, int dh, int f, int ra, int rm);
size_t lr_block_workspace_bytes(int b, int s, int H, int dh, int f, int ra, int rm);
lr_status lr_block_fwd(lr_dtype dt, int b, int s, int H, int dh, int f, int ra, int rm, float eps, const void* x,
                       const lr_block_weights* w, void* out, void* saved, size_t saved_bytes, void* ws,
                       size_t ws_bytes, void* stream);
lr_status lr_block_bwd(lr_dtype dt, int b, int s, int H, int dh, int f, int ra, int rm, float eps, const void* x,
                       const lr_block_weights* w, const void* saved, size_t saved_bytes, const void* dout, void* dx,
                       const lr_block_grads* g, void* ws, size_t ws_bytes, void* stream);

/* -------------------------------------------------------------- block stack
 * One training step of `nblocks` residual MLP blocks (as lr_mlp_fwd, sigma = SiLU) and a
 * mean-squared-error loss against `target` [T, d]:
 *     x_0 = x, x_{l+1} = block_l(x_l), loss = mean((x_L - target)^2)
 * then the backward through every block (in LR_SAVE_CKPT each block is
 * re-forwarded from its saved input and bottleneck pre-activations).
 * gs[l] is block l's gain [d]; pairs holds 3*nblocks pairs (gate, up, down of
 * block 0, then block 1, ...); dgs[l] [d] and grads (3*nblocks) receive the fp32
 * gradients; loss is a device fp32 scalar; dx [T,d] (dtype) may be NULL.
 * All activations of the step live in `ws`.
 */
size_t lr_stack_workspace_bytes(lr_dtype dt, lr_mode mode, int nblocks, int T, int d, int f, int r);

lr_status lr_stack_step(lr_dtype dt, lr_mode mode, int nblocks, int T, int d, int f, int r, float eps,
                        const void* x, const void* target, const void* const* gs, const lr_pair* pairs,
                        float* loss, void* dx, float* const* dgs, const lr_pair_grad* grads, void* ws,
                        size_t ws_bytes, void* stream);

/* ------------------------------------------------- allocation-free variant
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc — code running inside a framework whose
 * allocator owns all device memory, code under a memory budget that forbids
 * new allocations, or code paths that must not synchronise the device (as a
 * cudaMalloc/cudaFree can).  Such callers cannot provide `ws` for lr_proj_fwd.
 *
 * lr_proj_fwd_noalloc computes exactly what lr_proj_fwd (act = LR_ACT_SILU) computes, with the same
 * arguments minus the workspace.  Its only scratch (the gain-folded, stacked
 * A weights: group * r * d_in elements of the storage dtype) lives in one
 * file-scope device array of LR_NOALLOC_SCRATCH_BYTES bytes inside this
 * library; a call whose group * r * d_in * sizeof(dtype) exceeds it returns
 * LR_ERR_WORKSPACE and launches nothing.  The caller still allocates the inputs,
 * `outs` and `saved`.  The call allocates and frees nothing itself.
 *   - Every GPU that loads the library holds the array until the process exits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the array and it keeps the last call's contents (each
 *     call overwrites what it uses before reading it).  Calls that overlap on
 *     the GPU — on different streams, or from different host threads — race
 *     on it: serialise them.
 *   - It returns LR_ERR_UNSUPPORTED while profiling is on (the profiler
 *     creates CUDA events). */
#define LR_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
lr_status lr_proj_fwd_noalloc(lr_dtype dt, int T, int d_in, int d_out, int r, int group, const lr_pair* pairs,
                              const void* g, float eps, const void* x, void* const* outs, void* saved,
                              size_t saved_bytes, void* stream);

/* ------------------------------------------------------------------ status
 * lr_last_error: message of the last failing call on this thread ("" if none).
 * lr_check_device_error: synchronises `stream`, reads and clears the current
 * device's error word; LR_ERR_TIMEOUT if a bounded wait ran out, LR_ERR_CUDA
 * if the stream reports an error, else LR_OK.
 * lr_selftest_wait_timeout: launches one kernel that waits on a barrier nothing
 * completes, for limit_ns nanoseconds, then sets the timeout bit and returns
 * (exercises the timeout path without any fault). */
const char* lr_last_error(void);
lr_status lr_check_device_error(void* stream);
lr_status lr_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/* ------------------------------------------------------------- profiling
 * Instrumentation (no counterpart on the pages; it serves the measurement of
 * the path against its roofline).
 * lr_launch_count: kernels this library has launched in the process so far.
 * lr_profile_start: from now on bracket every launch by two CUDA events on its
 *   stream (clears earlier records).  lr_profile_stop: stop, synchronise the
 *   recorded events and aggregate them per kernel name.  Then entries
 *   0 .. lr_profile_count()-1 give each kernel's name, launches, total device
 *   milliseconds, and algorithmic FLOPs (GEMMs: 2 M N K per accumulator and
 *   batch entry) or bytes (memory-bound kernels) summed over its launches.
 * lr_profile_filter: record only launches whose kernel name starts with
 *   `prefix` (NULL or "" records all; the setting outlives start/stop).  Events
 *   between two launches end the overlap of the second one's start with the
 *   first one's tail, so a step timed under the profiler runs a little slower
 *   than one timed with events around the step alone. */
unsigned long long lr_launch_count(void);
lr_status lr_profile_start(void);
lr_status lr_profile_stop(void);
lr_status lr_profile_filter(const char* prefix);
int lr_profile_count(void);
lr_status lr_profile_entry(int i, char* name, size_t name_len, long long* launches, double* total_ms,
                           double* flops, double* bytes);

/* Library version (major * 10000 + minor * 100 + patch). */
int lr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LOWRANK_H_ */
