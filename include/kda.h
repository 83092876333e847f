/*
 * kda.h -- C ABI of the GB300-native chunk-parallel Kimi Delta Attention
 * (KDA) forward and backward library (libkda_gb300.so).
 *
 * The operation (kda_fwd, kda_bwd and kda_bwd_noalloc compute this operator;
 * kda_gdn2_fwd / kda_gdn2_bwd compute its GDN-2 generalisation, declared
 * further down; see the page "KDA Memory with Recompute: FLA vs cuDNN
 * Frontend FROST", section "Sources and measurement configuration", for the
 * operator configuration):
 *
 *   per packed sequence n (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1) and
 *   per head h, with state S (D x D; S_0 = h0[n][h], zero unless given; the
 *   final state S_T is returned as hT[n][h] when asked for):
 *     qh_t   = scale * q_t / sqrt(|q_t|^2 + l2_eps)
 *     kh_t   = k_t / sqrt(|k_t|^2 + l2_eps)
 *     beta_t = sigmoid(beta_raw_t)
 *     g_t    = gate_lower_bound * sigmoid(exp(A_log[h]) * (g_raw_t + dt_bias[h,:]))
 *     S_t    = (I - beta_t kh_t kh_t^T) Diag(exp(g_t)) S_{t-1} + beta_t kh_t v_t^T
 *     o_t    = S_t^T qh_t
 *   The gate's closed form is this library's reading of "safe gate with
 *   lower bound -5" built from the raw gate, A_log and dt_bias; the pages do
 *   not print it. The chunked evaluation (intra-chunk WY factors, serial
 *   inter-chunk state scan) follows "KDA at the production shape ...",
 *   section 2.1 (per-chunk op table) and section 1.1 (state scan).
 *
 * Layouts (all row-major, contiguous, no strides):
 *   q, k, v, g_raw, o, dO, dq, dk, dv, dg_raw : [S, H, D]  (token-major)
 *   beta_raw, dbeta_raw                        : [S, H]
 *   A_log, dA_log                              : [H]      fp32
 *   dt_bias, ddt_bias                          : [H, D]   fp32
 *   cu_seqlens                                 : [num_seqs + 1] int32, device
 *   h0, hT, dhT, dh0 (optional states)         : [num_seqs, H, D, D] fp32
 *   S = cu_seqlens[num_seqs] = total_tokens; K = V = D = head_dim.
 *   Element type of the [S,H,D] and [S,H] tensors is problem->dtype.
 *
 * Ownership: the caller allocates every buffer (inputs, outputs, ctx,
 * workspace) in device memory. The library never allocates or frees device
 * memory, never synchronises the stream inside kda_fwd / kda_bwd, and keeps
 * no pointer after a call returns. Outputs are overwritten (=), never
 * accumulated. Inputs are read-only. Outputs must not alias inputs.
 *
 * Errors: every entry point validates its arguments on the host and returns
 * a kda_status without launching anything when they are bad. Launch failures
 * map to KDA_ERR_CUDA. Errors detected inside a kernel (a bounded wait that
 * ran out, a failed device-side check) are written to a status word inside
 * ctx (forward) or workspace (backward) and read with
 * kda_query_device_status. Kernels never trap.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream). All device work of a call is enqueued on that stream.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  KDA_ERR_UNSUPPORTED = 2,   /* head_dim / dtype combination not built */
  KDA_ERR_WORKSPACE = 3,     /* ctx or workspace smaller than required */
  KDA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  KDA_ERR_TIMEOUT = 5,       /* device side: a bounded wait ran out */
  KDA_ERR_DEVICE_CHECK = 6   /* device side: an in-kernel check failed */
} kda_status;

typedef enum {
  KDA_DTYPE_BF16 = 0,
  KDA_DTYPE_F32 = 1
} kda_dtype;

/* kda_problem.flags bits. KDA_FLAG_FORCE_SIMT runs the fp32 CUDA-core
 * kernels even where tensor-core kernels exist (bf16, head_dim 128): slower,
 * fp32 accuracy throughout. */
#define KDA_FLAG_FORCE_SIMT 1
/* Test only: exercises the device-side failure path without faulting the GPU.
 * The tensor-core forward skips the first q/k/gate tile load, so its bounded
 * wait for that load runs out (after a short spin); the kernel records
 * KDA_ERR_TIMEOUT in ctx's status word, frees its tensor memory and returns.
 * o is not written. kda_query_device_status(ctx) then reports the timeout and
 * the context stays usable. Ignored by the CUDA-core kernels. */
#define KDA_FLAG_TEST_TIMEOUT 2
/* Inference: kda_fwd writes no state checkpoints. ctx (optional, of
 * kda_ctx_bytes(p) bytes with this flag set, which leaves the checkpoints
 * out) then only holds the status word and, when the tensor-core forward
 * runs with helper CTAs, their hand-off area, so the forward keeps that
 * speed-up without a checkpoint buffer. Such a ctx cannot feed kda_bwd, which
 * rejects the flag. */
#define KDA_FLAG_NO_CHECKPOINTS 4
/* GDN-2 problem: the operator with channel-wise erase and write gates
 * (kda_gdn2_fwd / kda_gdn2_bwd below). Set it before the size queries so
 * that they size ctx and workspace for the GDN-2 kernels; kda_fwd, kda_bwd
 * and kda_bwd_noalloc reject it, and kda_gdn2_fwd / kda_gdn2_bwd require it.
 * The GDN-2 forward runs on the tensor-core kernels for bf16 with head_dim
 * 128 (the CUDA-core kernels otherwise); the GDN-2 backward runs on the
 * fp32 CUDA-core kernels for every dtype and head_dim. */
#define KDA_FLAG_CHANNEL_GATES 8
/* kda_fwd with 16-token chunks ("KDA at the production shape ...", section
 * 1.3: the chunk size of the FlashKDA and FLA forwards it compares) instead
 * of the default 64-token chunks with 16-token sub-block references. It runs
 * on the tensor cores for bf16 with head_dim 128 (KDA_ERR_UNSUPPORTED for
 * other problems, with KDA_FLAG_FORCE_SIMT, or for GDN-2): one CTA per
 * (sequence, head) at a time walks the chunks in order, with O = (Qh Gamma) H
 * + M U~ per chunk, and stores the same checkpoints as the default forward
 * (none with KDA_FLAG_NO_CHECKPOINTS), so its ctx feeds kda_bwd. Same outputs
 * to within rounding. kda_bwd ignores the flag. */
#define KDA_FLAG_CHUNK16 16

/* Problem description. cu_seqlens is a DEVICE pointer; the library never
 * reads it on the host (so no synchronisation). It must start at 0, be
 * non-decreasing and end at total_tokens. Every call checks this on the
 * device before its kernels run: a one-CTA kernel copies cu_seqlens into the
 * call's own buffer (after the 256-byte header of ctx for the forward, of
 * workspace for the backward, of the library's array for kda_bwd_noalloc),
 * and the kernels read only that copy. If any of the three conditions fails,
 * the copy is all zeros instead, so every sequence is empty and no kernel
 * indexes inputs, outputs, checkpoints or scratch through the malformed
 * array, and KDA_ERR_DEVICE_CHECK is recorded in the call's status word
 * (kda_query_device_status / kda_noalloc_device_status). The call then
 * writes no o or activation gradient; hT = h0, dh0 = dhT, dA_log = ddt_bias
 * = 0. A forward given ctx == NULL has neither a status word nor a buffer
 * for the copy: it reads cu_seqlens unchecked. */
typedef struct {
  int64_t total_tokens;       /* S */
  int32_t num_seqs;           /* N >= 1 */
  int32_t num_heads;          /* H >= 1 */
  int32_t head_dim;           /* D = K = V; 64 or 128 */
  int32_t dtype;              /* kda_dtype of the [S,H,D] / [S,H] tensors */
  float scale;                /* output scale applied to qh (1.0 = none) */
  float gate_lower_bound;     /* L < 0, e.g. -5.0 */
  float l2_eps;               /* epsilon inside the L2-norm square root */
  int32_t flags;              /* KDA_FLAG_* bits, 0 by default */
  const int32_t* cu_seqlens;  /* device, num_seqs + 1 entries */
} kda_problem;

/* Bytes of the forward->backward context: a 256-byte header holding the
 * forward's device status word, the checked copy of cu_seqlens (num_seqs + 1
 * int32, rounded up to 256 bytes), then the state checkpoints (fp32, one per
 * 1024 tokens of every sequence and head). Returns 0 for an invalid problem. The size
 * queries ignore cu_seqlens (it may be NULL). */
size_t kda_ctx_bytes(const kda_problem* p);

/* Bytes of the backward workspace: a 256-byte header with the backward's
 * device status word, the checked copy of cu_seqlens, gate-parameter partial
 * sums and scratch for the recomputed chunk states of checkpoint segments. Returns 0 for an
 * invalid problem. */
size_t kda_bwd_workspace_bytes(const kda_problem* p);

/* Recurrent states at the ABI (initial state h0, final state hT and their
 * gradients dh0, dhT): fp32 [N][H][D][D], contiguous, row index = key
 * channel i, column index = value channel j, so that one sequence's state is
 * the D x V matrix S of the recurrence. Every state pointer is optional:
 * NULL h0 / dhT mean zero, NULL hT / dh0 are not written.
 * On the tensor-core backward, when dhT is given or dh0 asked for, the gate
 * gradient of each sequence's first and last chunk uses the chunk-start
 * state to fp32 accuracy (there h0 or dhT meet it in one product); without
 * either, those chunks use the same fp16 state operand as the others, which
 * is exact when h0 is zero. A caller that starts the forward from h0 should
 * therefore ask the backward for dh0. */

/* Forward. Writes o [S,H,D] and, when hT is not NULL, the final states;
 * the recurrence of sequence n, head h starts from h0[n][h] (zero when h0 is
 * NULL). When ctx is not NULL it must hold kda_ctx_bytes(p) bytes (16-byte
 * aligned); the forward writes the state checkpoints there for kda_bwd, and
 * ctx must then stay alive and unmodified until the matching kda_bwd has been
 * enqueued. ctx == NULL runs the forward alone (inference), writing no
 * checkpoints. All tensor pointers must be 16-byte aligned. */
kda_status kda_fwd(const kda_problem* p,
                   const void* q, const void* k, const void* v,
                   const void* g_raw, const void* beta_raw,
                   const float* A_log, const float* dt_bias,
                   const float* h0,
                   void* o, float* hT, void* ctx, void* stream);

/* Backward. Given dO [S,H,D], the gradient of the final states dhT (zero
 * when NULL) and the ctx written by kda_fwd on the same inputs (and the same
 * h0: the checkpoints carry it), writes dq, dk, dv, dg_raw [S,H,D],
 * dbeta_raw [S,H] (problem dtype), dA_log [H], ddt_bias [H,D] (fp32) and,
 * when dh0 is not NULL, the gradient of the initial states. It recomputes
 * the chunk states, the WY factors and the gated q/k chunk by chunk from the
 * inputs and the checkpoints; no full-sequence intermediate is stored.
 * workspace must hold kda_bwd_workspace_bytes(p) bytes (16-byte aligned). */
kda_status kda_bwd(const kda_problem* p,
                   const void* q, const void* k, const void* v,
                   const void* g_raw, const void* beta_raw,
                   const float* A_log, const float* dt_bias,
                   const void* dO, const float* dhT, const void* ctx,
                   void* dq, void* dk, void* dv, void* dg_raw, void* dbeta_raw,
                   float* dA_log, float* ddt_bias, float* dh0,
                   void* workspace, void* stream);

/* Size of the fixed scratch buffer that kda_bwd_noalloc uses (64 MiB). */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* Backward without any device allocation. The paper has no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc where they run
 * the backward (a host that serves all device memory from its own fixed
 * pool, a plug-in handed device pointers but no allocator, a loop that must
 * not take an allocation's implicit synchronisation). Same arguments,
 * layouts and results as kda_bwd, minus the workspace: the backward's scratch
 * (gate-parameter partials and recomputed chunk-start states) lives in a
 * KDA_NOALLOC_SCRATCH_BYTES array inside the library, which every GPU that
 * loads the library holds until the process exits. The caller still passes
 * all inputs and outputs. It calls no cudaMalloc / cudaFree and no
 * allocating library routine.
 * - The first call on a device looks up that device's address of the array
 *   (cudaGetSymbolAddress, with the device current); make that first call
 *   before any stream capture.
 * - Problems whose scratch does not fit (header + partials for N*H
 *   sequence-heads + one CTA's segment states) return KDA_ERR_WORKSPACE
 *   with the required size in kda_last_error_message(); use kda_bwd then.
 * - It runs the same kernel family as kda_bwd (kda_kernel_family), so the
 *   two give bit-identical results; fewer CTAs fit than kda_bwd would use,
 *   so it is slower.
 * - Every call shares the array: calls whose GPU work overlaps (other
 *   streams or threads on the same device) race and give wrong results.
 * - Its device-side status word (a bounded wait that ran out, a malformed
 *   cu_seqlens) sits in the array: read it with kda_noalloc_device_status. */
kda_status kda_bwd_noalloc(const kda_problem* p,
                           const void* q, const void* k, const void* v,
                           const void* g_raw, const void* beta_raw,
                           const float* A_log, const float* dt_bias,
                           const void* dO, const float* dhT, const void* ctx,
                           void* dq, void* dk, void* dv, void* dg_raw, void* dbeta_raw,
                           float* dA_log, float* ddt_bias, float* dh0, void* stream);

/* Device status word of the last kda_bwd_noalloc call on the current
 * device (the word at the head of the library's fixed scratch array),
 * copied into a host int without any allocation. Synchronises `stream`
 * first. Returns KDA_OK, KDA_ERR_TIMEOUT or KDA_ERR_DEVICE_CHECK as recorded
 * by the kernels, or KDA_ERR_CUDA if the read failed. The paper has no
 * counterpart: it completes the no-allocation entry point above. */
kda_status kda_noalloc_device_status(void* stream);

/* GDN-2: the same operator with the scalar beta replaced by two channel-wise
 * gates ("KDA at the production shape ...", section 1.6, which names GDN-2
 * as this generalisation with KDA its special case, and the section 2.1 op
 * table: akk = (b*k*Gamma)(k/Gamma)^T, w = M^-1 (b k*Gamma), u = M^-1 (w*v)):
 *     b_t = sigmoid(erase_raw_t)   (per key channel)
 *     w_t = sigmoid(write_raw_t)   (per value channel)
 *     S_t = (I - kh_t (b_t * kh_t)^T) Diag(exp(g_t)) S_{t-1} + kh_t (w_t * v_t)^T
 *     o_t = S_t^T qh_t
 * with qh, kh, g, scale, states and sequence packing exactly as for KDA
 * (b_t = w_t = beta_t on every channel gives KDA). The sigmoid of the two raw
 * gates mirrors beta's; the pages print no activation for them.
 * erase_raw, write_raw, derase_raw, dwrite_raw: [S, H, D] in problem->dtype.
 * p->flags must include KDA_FLAG_CHANNEL_GATES (KDA_ERR_INVALID_ARG
 * otherwise), and ctx / workspace must then hold kda_ctx_bytes(p) /
 * kda_bwd_workspace_bytes(p) bytes of that problem. Every other argument,
 * ownership rule and error behaviour is that of kda_fwd / kda_bwd;
 * KDA_FLAG_NO_CHECKPOINTS works as for kda_fwd. */
kda_status kda_gdn2_fwd(const kda_problem* p,
                        const void* q, const void* k, const void* v,
                        const void* g_raw, const void* erase_raw, const void* write_raw,
                        const float* A_log, const float* dt_bias,
                        const float* h0,
                        void* o, float* hT, void* ctx, void* stream);

kda_status kda_gdn2_bwd(const kda_problem* p,
                        const void* q, const void* k, const void* v,
                        const void* g_raw, const void* erase_raw, const void* write_raw,
                        const float* A_log, const float* dt_bias,
                        const void* dO, const float* dhT, const void* ctx,
                        void* dq, void* dk, void* dv, void* dg_raw,
                        void* derase_raw, void* dwrite_raw,
                        float* dA_log, float* ddt_bias, float* dh0,
                        void* workspace, void* stream);

/* Affine state prefix: the exchange step that joins the pieces of sequences
 * cut in time (context parallelism). The recurrence is linear in its state,
 * so for fixed inputs piece p of a sequence maps its start state to its end
 * state affinely, H_end = A_p H_start + B_p (A_p: D x D on the key index;
 * it is the piece's final state when the piece runs from the identity state
 * with zero values, B_p the final state when it runs from zero with its
 * values, both from kda_fwd with hT; GDN-2's recurrence is affine in its
 * state in the same way, so kda_gdn2_fwd / kda_gdn2_bwd give its maps). The
 * backward is the transposed map: a
 * piece's start-state gradient is A_p^T (its end-state gradient) + C_p,
 * with C_p the dh0 of the piece's kda_bwd run with dhT = 0. Given every
 * piece's (A_p, B_p) or (A_p, C_p), this prefix returns each piece's true
 * start state (forward) or true end-state gradient (backward); the pieces
 * then run kda_fwd / kda_bwd independently with those h0 / dhT, on one GPU
 * (the pieces packed as sequences of one launch) or one piece per GPU after
 * the maps have been gathered from the ranks. The pages measure no such
 * split ("KDA Memory with Recompute ...", section "Measured peak allocated
 * memory", leaves every 256K-token case unmeasured); the algebra is the
 * state recurrence's own.
 *   num_seqs N, pieces P >= 1, num_heads H, head_dim D (64 or 128).
 *   A, B, xs: fp32 D x D matrices; the one of (piece p, sequence n, head h)
 *     starts at element (p * piece_stride + n * seq_stride + h) * D * D.
 *     piece_stride = H, seq_stride = P * H is the layout kda_fwd / kda_bwd
 *     give when each sequence's P pieces are packed as P consecutive
 *     sequences ([N][P][H][D][D]); piece_stride = N * H, seq_stride = H is
 *     the layout of maps gathered from P ranks ([P][N][H][D][D]). Padded
 *     strides are accepted as long as the matrices cannot overlap: either
 *     piece_stride >= H and seq_stride >= P * piece_stride, or
 *     seq_stride >= H and piece_stride >= N * seq_stride. Any other pair
 *     returns KDA_ERR_INVALID_ARG.
 *   x0, x_end: fp32 [N][H][D][D].
 *   KDA_PREFIX_FORWARD:  x_0 = x0 (zero when NULL), xs[p] = x_p,
 *                        x_{p+1} = A_p x_p + B_p, x_end = x_P (if not NULL).
 *   KDA_PREFIX_BACKWARD: x_{P-1} = x0 (zero when NULL), xs[p] = x_p,
 *                        x_{p-1} = A_p^T x_p + B_p, x_end = A_0^T x_0 + B_0.
 * Device pointers, 16-byte aligned; fp32 accumulation; asynchronous on
 * `stream`; one CTA per (sequence, head). Returns KDA_ERR_INVALID_ARG /
 * KDA_ERR_UNSUPPORTED for bad arguments, KDA_ERR_CUDA if the launch fails. */
#define KDA_PREFIX_FORWARD 0
#define KDA_PREFIX_BACKWARD 1
kda_status kda_state_prefix(int32_t num_seqs, int32_t pieces, int32_t num_heads, int32_t head_dim,
                            int32_t direction, int64_t piece_stride, int64_t seq_stride,
                            const float* A, const float* B, const float* x0, float* xs, float* x_end,
                            void* stream);

/* Reads the device status word at the head of a ctx or workspace buffer.
 * Synchronises `stream` first. Returns KDA_OK, KDA_ERR_TIMEOUT or
 * KDA_ERR_DEVICE_CHECK as recorded by the kernels, or KDA_ERR_CUDA if the
 * read itself failed. */
kda_status kda_query_device_status(const void* ctx_or_workspace, void* stream);

/* Static, NUL-terminated name of a status code. */
const char* kda_status_string(kda_status s);

/* Detail of the last error returned on the calling thread (static storage,
 * overwritten by the next failing call on that thread). */
const char* kda_last_error_message(void);

/* Which kernel families a problem's forward and backward dispatch to: 0 =
 * fp32 CUDA-core (SIMT) kernels for both, 1 = tcgen05 tensor-core kernels
 * for both (bf16, head_dim 128, unless KDA_FLAG_FORCE_SIMT), 2 = tensor-core
 * forward and CUDA-core backward (GDN-2 problems in bf16 with head_dim 128);
 * -1 for an invalid or unsupported problem. Host only. */
int kda_kernel_family(const kda_problem* p);

/* Library ABI version, major * 100 + minor * 10 (230 = 2.3: KDA_FLAG_CHUNK16; 220 = 2.2: the affine state prefix,
 * the no-allocation status query and the device-side cu_seqlens check). */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
