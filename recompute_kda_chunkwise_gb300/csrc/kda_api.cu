// kda_api.cu -- host side of the C ABI declared in include/kda.h: argument
// validation, buffer sizing, kernel-family dispatch and launches. No device
// memory is allocated here and no stream is synchronised inside kda_fwd /
// kda_bwd.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "kda_internal.cuh"

namespace {

thread_local char g_msg[512] = "";

kda_status fail(kda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Largest |lower bound| for which the chunk-factored intra products stay in
// fp32 range: |L| * 16 tokens * log2(e) must stay below 128 binary orders.
constexpr float kMaxAbsLower = 5.5f;

kda_status validate(const kda_problem* p, bool need_ptrs = true) {
  if (!p) return fail(KDA_ERR_INVALID_ARG, "problem is NULL");
  if (p->num_seqs < 1) return fail(KDA_ERR_INVALID_ARG, "num_seqs must be >= 1 (got %d)", p->num_seqs);
  if (p->num_heads < 1) return fail(KDA_ERR_INVALID_ARG, "num_heads must be >= 1 (got %d)", p->num_heads);
  if (p->total_tokens < 0) return fail(KDA_ERR_INVALID_ARG, "total_tokens must be >= 0");
  if ((p->flags & ~(KDA_FLAG_FORCE_SIMT | KDA_FLAG_TEST_TIMEOUT | KDA_FLAG_NO_CHECKPOINTS |
                    KDA_FLAG_CHANNEL_GATES | KDA_FLAG_CHUNK16)) != 0)
    return fail(KDA_ERR_INVALID_ARG, "unknown flags 0x%x", p->flags);
  if (need_ptrs && !p->cu_seqlens) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (p->dtype != KDA_DTYPE_BF16 && p->dtype != KDA_DTYPE_F32)
    return fail(KDA_ERR_UNSUPPORTED, "dtype %d is not supported", p->dtype);
  if (p->head_dim != 64 && p->head_dim != 128)
    return fail(KDA_ERR_UNSUPPORTED, "head_dim %d is not supported (64 or 128)", p->head_dim);
  if (!isfinite(p->scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
  if (!(p->l2_eps >= 0.f) || !isfinite(p->l2_eps)) return fail(KDA_ERR_INVALID_ARG, "l2_eps must be >= 0");
  if (!(p->gate_lower_bound <= 0.f) || p->gate_lower_bound < -kMaxAbsLower)
    return fail(KDA_ERR_UNSUPPORTED, "gate_lower_bound must lie in [-%.1f, 0] (got %g)", kMaxAbsLower,
                p->gate_lower_bound);
  // element counts must fit comfortably in int64 offsets
  if (p->total_tokens > ((int64_t)1 << 40) / ((int64_t)p->num_heads * p->head_dim))
    return fail(KDA_ERR_INVALID_ARG, "problem too large");
  if ((int64_t)p->num_seqs * p->num_heads > (1 << 30)) return fail(KDA_ERR_INVALID_ARG, "too many sequences x heads");
  return KDA_OK;
}

// Kernel family of each pass: tcgen05 kernels for bf16 D = 128 (unless
// KDA_FLAG_FORCE_SIMT), else fp32 SIMT. GDN-2 problems (channel-wise gates)
// run the tensor-core forward but the SIMT backward.
int fwd_family_of(const kda_problem* p) {
  return (p->dtype == KDA_DTYPE_BF16 && p->head_dim == 128 && !(p->flags & KDA_FLAG_FORCE_SIMT)) ? 1 : 0;
}
int family_of(const kda_problem* p) {  // the backward's
  return (fwd_family_of(p) == 1 && !(p->flags & KDA_FLAG_CHANNEL_GATES)) ? 1 : 0;
}

size_t ckpt_slots(const kda_problem* p) {
  return (size_t)(p->total_tokens / kda::kCkptTokens) + (size_t)p->num_seqs;
}

size_t ckpt_bytes(const kda_problem* p) {
  if (p->flags & KDA_FLAG_NO_CHECKPOINTS) return 0;
  const size_t D = (size_t)p->head_dim;
  return ckpt_slots(p) * (size_t)p->num_heads * D * D * sizeof(float);
}

// Tensor-core forward with fewer (sequence, head) items than the 152-CTA
// grid: the spare SMs prepare every other chunk; the hand-off area follows
// the checkpoints in ctx.
size_t fwd_handoff(const kda_problem* p) {
  const int64_t items = (int64_t)p->num_seqs * p->num_heads;
  if (fwd_family_of(p) != 1 || items <= 0 || items >= kda::kTcBwdCtas) return 0;
  return kda::fwd_handoff_bytes((int)items);
}

size_t cu_bytes(const kda_problem* p) { return kda::cu_copy_bytes(p->num_seqs); }

size_t ctx_bytes(const kda_problem* p) { return kda::kHeaderBytes + cu_bytes(p) + ckpt_bytes(p) + fwd_handoff(p); }

size_t partial_bytes(const kda_problem* p) {
  return round_up((size_t)p->num_seqs * p->num_heads * (p->head_dim + 1) * sizeof(float), 256);
}

int tc_bwd_ctas(const kda_problem* p) {
  const int64_t items = (int64_t)p->num_seqs * p->num_heads;
  return (int)(items < kda::kTcBwdCtas ? items : kda::kTcBwdCtas);
}

// Tensor-core backward: per-item hand-off counters for helper CTAs and their
// job counter (only problems with fewer items than the 152-CTA grid use them).
size_t flag_bytes(const kda_problem* p) {
  if (family_of(p) != 1) return 0;
  return round_up(((size_t)tc_bwd_ctas(p) * kda::kTcBwdFlags + 1) * sizeof(uint32_t), 256);
}

// Tensor-core backward: per-item low parts of the sequence-edge chunk states.
size_t edge_bytes(const kda_problem* p) {
  if (family_of(p) != 1) return 0;
  return kda::bwd_edge_bytes_tc((int64_t)p->num_seqs * p->num_heads);
}

size_t workspace_bytes(const kda_problem* p) {
  size_t scratch = kda::bwd_scratch_bytes_simt(p, nullptr);
  if (family_of(p) == 1) {
    // inline mode: one segment's states per CTA; split mode (items < 152):
    // kTcBwdBufs segment buffers per item
    const int64_t items = (int64_t)p->num_seqs * p->num_heads;
    scratch = edge_bytes(p) +
              (items < kda::kTcBwdCtas ? (size_t)items * kda::kTcBwdBufs * kda::bwd_scratch_bytes_per_buf_split_tc()
                                       : (size_t)kda::kTcBwdCtas * kda::bwd_scratch_bytes_per_cta_tc());
  }
  return kda::kHeaderBytes + cu_bytes(p) + partial_bytes(p) + flag_bytes(p) + scratch;
}

#define CHECK_PTR(ptr)                                                                   \
  do {                                                                                   \
    if (!(ptr)) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", #ptr);                    \
    if (!aligned16(ptr)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #ptr); \
  } while (0)
#define CHECK_OPT(ptr)                                                                             \
  do {                                                                                             \
    if ((ptr) && !aligned16(ptr)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #ptr); \
  } while (0)

// Bytes of one [N][H][D][D] fp32 state tensor.
size_t state_bytes(const kda_problem* p) {
  return (size_t)p->num_seqs * p->num_heads * p->head_dim * p->head_dim * sizeof(float);
}

// dst = src (or zero when src is NULL): the state of a sequence without tokens.
kda_status pass_state(float* dst, const float* src, const kda_problem* p, cudaStream_t s) {
  if (!dst) return KDA_OK;
  const cudaError_t e = src ? cudaMemcpyAsync(dst, src, state_bytes(p), cudaMemcpyDeviceToDevice, s)
                            : cudaMemsetAsync(dst, 0, state_bytes(p), s);
  return e == cudaSuccess ? KDA_OK
                          : fail(KDA_ERR_CUDA, "state copy failed: %s", cudaGetErrorString(cudaGetLastError()));
}

}  // namespace

namespace kda {

namespace {
// One CTA: cu_out = cu if cu[0] == 0, cu is non-decreasing and cu[N] == S,
// else all zeros (every sequence empty, so no kernel indexes anything
// through the malformed array) and KDA_ERR_DEVICE_CHECK in *status.
__global__ void __launch_bounds__(256) kda_check_cu_kernel(const int32_t* cu, int N, int64_t S, int32_t* cu_out,
                                                          int* status) {
  int bad = 0;
  for (int i = static_cast<int>(threadIdx.x); i <= N; i += static_cast<int>(blockDim.x)) {
    const int64_t c = cu[i];
    if (i == 0 && c != 0) bad = 1;
    if (i > 0 && c < static_cast<int64_t>(cu[i - 1])) bad = 1;
    if (c < 0 || c > S || (i == N && c != S)) bad = 1;
  }
  bad = __syncthreads_or(bad);
  for (int i = static_cast<int>(threadIdx.x); i <= N; i += static_cast<int>(blockDim.x)) cu_out[i] = bad ? 0 : cu[i];
  if (bad && threadIdx.x == 0) set_status(status, KDA_ERR_DEVICE_CHECK);
}
}  // namespace

kda_status launch_check_cu(const int32_t* cu, int N, int64_t S, int32_t* cu_out, int* status, cudaStream_t s) {
  kda_check_cu_kernel<<<1, 256, 0, s>>>(cu, N, S, cu_out, status);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status validate_problem(const kda_problem* p) { return validate(p); }
kda_status set_error(kda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}
size_t gate_partial_bytes(const kda_problem* p) { return partial_bytes(p); }
int kernel_family(const kda_problem* p) { return family_of(p); }
}  // namespace kda

extern "C" {

size_t kda_ctx_bytes(const kda_problem* p) { return validate(p, false) == KDA_OK ? ctx_bytes(p) : 0; }

size_t kda_bwd_workspace_bytes(const kda_problem* p) {
  return validate(p, false) == KDA_OK ? workspace_bytes(p) : 0;
}

int kda_kernel_family(const kda_problem* p) {
  if (validate(p, false) != KDA_OK) return -1;
  return fwd_family_of(p) == family_of(p) ? family_of(p) : 2;
}

int kda_version(void) { return 230; }

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK";
  }
  return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error_message(void) { return g_msg; }

}  // extern "C"

namespace {

// Forward of both operators: write_raw is NULL for KDA (beta_raw [S,H]) and
// set for GDN-2 (beta_raw is then the erase gate [S,H,D]).
kda_status forward(const kda_problem* p, const void* q, const void* k, const void* v, const void* g_raw,
                   const void* beta_raw, const void* write_raw, const float* A_log, const float* dt_bias,
                   const float* h0, void* o, float* hT, void* ctx, void* stream) {
  kda_status st = validate(p);
  if (st != KDA_OK) return st;
  CHECK_OPT(h0); CHECK_OPT(hT);
  // 16-token chunks: tensor-core KDA problems only (refused before any launch)
  if ((p->flags & KDA_FLAG_CHUNK16) && (fwd_family_of(p) != 1 || write_raw != nullptr))
    return fail(KDA_ERR_UNSUPPORTED, "KDA_FLAG_CHUNK16 needs a KDA problem in bf16 with head_dim 128");
  if (p->total_tokens == 0) return pass_state(hT, h0, p, (cudaStream_t)stream);  // hT = h0
  CHECK_PTR(q); CHECK_PTR(k); CHECK_PTR(v); CHECK_PTR(g_raw); CHECK_PTR(beta_raw);
  CHECK_PTR(A_log); CHECK_PTR(dt_bias); CHECK_PTR(o);
  if (ctx && !aligned16(ctx)) return fail(KDA_ERR_INVALID_ARG, "ctx is not 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  kda::FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g_raw; a.b = beta_raw; a.A_log = A_log; a.dt_bias = dt_bias;
  a.o = o;
  a.h0 = h0;
  a.hT = hT;
  char* after_cu = ctx ? (char*)ctx + kda::kHeaderBytes + cu_bytes(p) : nullptr;
  a.ckpt = (ctx && ckpt_bytes(p)) ? (float*)after_cu : nullptr;
  a.status = ctx ? (int*)ctx : nullptr;
  // with a ctx the kernels read the checked copy of cu_seqlens kept in it
  a.cu = ctx ? (const int32_t*)((char*)ctx + kda::kHeaderBytes) : p->cu_seqlens;
  a.S = p->total_tokens; a.N = p->num_seqs; a.H = p->num_heads;
  a.scale = p->scale; a.lower = p->gate_lower_bound; a.eps = p->l2_eps;
  a.test_timeout = (p->flags & KDA_FLAG_TEST_TIMEOUT) ? 1 : 0;
  a.xflags = nullptr;
  a.xbuf = nullptr;
  a.w = write_raw;
  if (ctx && fwd_handoff(p)) {
    a.xflags = (uint32_t*)(after_cu + ckpt_bytes(p));
    a.xbuf = (uint8_t*)a.xflags + round_up((size_t)p->num_seqs * p->num_heads * 5 * sizeof(uint32_t), 256);
  }
  if (ctx && cudaMemsetAsync(ctx, 0, sizeof(int), s) != cudaSuccess)
    return fail(KDA_ERR_CUDA, "status reset failed: %s", cudaGetErrorString(cudaGetLastError()));
  if (ctx) {
    st = kda::launch_check_cu(p->cu_seqlens, p->num_seqs, p->total_tokens, (int32_t*)a.cu, a.status, s);
    if (st != KDA_OK) return fail(st, "cu_seqlens check launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  }
  if (p->flags & KDA_FLAG_CHUNK16)
    st = kda::launch_fwd16_tc(p, a, s);
  else
    st = fwd_family_of(p) == 1 ? kda::launch_fwd_tc(p, a, s) : kda::launch_fwd_simt(p, a, s);
  if (st != KDA_OK) return fail(st, "forward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return KDA_OK;
}

// Backward of both operators: write_raw / dwrite_raw are NULL for KDA and set
// for GDN-2 (beta_raw / dbeta_raw are then the erase gate and its gradient).
kda_status backward(const kda_problem* p, const void* q, const void* k, const void* v, const void* g_raw,
                    const void* beta_raw, const void* write_raw, const float* A_log, const float* dt_bias,
                    const void* dO, const float* dhT, const void* ctx, void* dq, void* dk, void* dv,
                    void* dg_raw, void* dbeta_raw, void* dwrite_raw, float* dA_log, float* ddt_bias,
                    float* dh0, void* workspace, void* stream) {
  kda_status st = validate(p);
  if (st != KDA_OK) return st;
  CHECK_OPT(dhT); CHECK_OPT(dh0);
  if (p->flags & KDA_FLAG_NO_CHECKPOINTS)
    return fail(KDA_ERR_INVALID_ARG, "KDA_FLAG_NO_CHECKPOINTS: a forward without checkpoints cannot feed kda_bwd");
  cudaStream_t s = (cudaStream_t)stream;
  if (p->total_tokens == 0) {  // no tokens: zero parameter gradients, dh0 = dhT
    CHECK_PTR(dA_log); CHECK_PTR(ddt_bias);
    if (cudaMemsetAsync(dA_log, 0, sizeof(float) * p->num_heads, s) != cudaSuccess ||
        cudaMemsetAsync(ddt_bias, 0, sizeof(float) * p->num_heads * p->head_dim, s) != cudaSuccess)
      return fail(KDA_ERR_CUDA, "memset failed: %s", cudaGetErrorString(cudaGetLastError()));
    return pass_state(dh0, dhT, p, s);
  }
  CHECK_PTR(q); CHECK_PTR(k); CHECK_PTR(v); CHECK_PTR(g_raw); CHECK_PTR(beta_raw);
  CHECK_PTR(A_log); CHECK_PTR(dt_bias); CHECK_PTR(dO); CHECK_PTR(ctx);
  CHECK_PTR(dq); CHECK_PTR(dk); CHECK_PTR(dv); CHECK_PTR(dg_raw); CHECK_PTR(dbeta_raw);
  CHECK_PTR(dA_log); CHECK_PTR(ddt_bias); CHECK_PTR(workspace);
  kda::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g_raw; a.b = beta_raw; a.A_log = A_log; a.dt_bias = dt_bias;
  a.dO = dO;
  a.dhT = dhT;
  a.dh0 = dh0;
  a.ckpt = (const float*)((const char*)ctx + kda::kHeaderBytes + cu_bytes(p));
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg_raw; a.db = dbeta_raw;
  a.dA_log = dA_log; a.ddt_bias = ddt_bias;
  a.status = (int*)workspace;
  char* ws = (char*)workspace + kda::kHeaderBytes;  // checked copy of cu_seqlens, then the rest
  a.partial = (float*)(ws + cu_bytes(p));
  a.flags = flag_bytes(p) ? (uint32_t*)(ws + cu_bytes(p) + partial_bytes(p)) : nullptr;
  a.edge = ws + cu_bytes(p) + partial_bytes(p) + flag_bytes(p);
  a.scratch = (float*)((char*)a.edge + edge_bytes(p));
  a.cu = (const int32_t*)ws;
  a.S = p->total_tokens; a.N = p->num_seqs; a.H = p->num_heads;
  a.scale = p->scale; a.lower = p->gate_lower_bound; a.eps = p->l2_eps;
  a.w = write_raw;
  a.dw = dwrite_raw;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess)
    return fail(KDA_ERR_CUDA, "status reset failed: %s", cudaGetErrorString(cudaGetLastError()));
  st = kda::launch_check_cu(p->cu_seqlens, p->num_seqs, p->total_tokens, (int32_t*)a.cu, a.status, s);
  if (st != KDA_OK) return fail(st, "cu_seqlens check launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  st = family_of(p) == 1 ? kda::launch_bwd_tc(p, a, s, tc_bwd_ctas(p)) : kda::launch_bwd_simt(p, a, s);
  if (st != KDA_OK) return fail(st, "backward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_fwd(const kda_problem* p, const void* q, const void* k, const void* v, const void* g_raw,
                   const void* beta_raw, const float* A_log, const float* dt_bias, const float* h0, void* o,
                   float* hT, void* ctx, void* stream) {
  if (p && (p->flags & KDA_FLAG_CHANNEL_GATES))
    return fail(KDA_ERR_INVALID_ARG, "KDA_FLAG_CHANNEL_GATES: a GDN-2 problem runs through kda_gdn2_fwd");
  return forward(p, q, k, v, g_raw, beta_raw, nullptr, A_log, dt_bias, h0, o, hT, ctx, stream);
}

kda_status kda_bwd(const kda_problem* p, const void* q, const void* k, const void* v, const void* g_raw,
                   const void* beta_raw, const float* A_log, const float* dt_bias, const void* dO,
                   const float* dhT, const void* ctx, void* dq, void* dk, void* dv, void* dg_raw,
                   void* dbeta_raw, float* dA_log, float* ddt_bias, float* dh0, void* workspace,
                   void* stream) {
  if (p && (p->flags & KDA_FLAG_CHANNEL_GATES))
    return fail(KDA_ERR_INVALID_ARG, "KDA_FLAG_CHANNEL_GATES: a GDN-2 problem runs through kda_gdn2_bwd");
  return backward(p, q, k, v, g_raw, beta_raw, nullptr, A_log, dt_bias, dO, dhT, ctx, dq, dk, dv, dg_raw,
                  dbeta_raw, nullptr, dA_log, ddt_bias, dh0, workspace, stream);
}

kda_status kda_gdn2_fwd(const kda_problem* p, const void* q, const void* k, const void* v, const void* g_raw,
                        const void* erase_raw, const void* write_raw, const float* A_log, const float* dt_bias,
                        const float* h0, void* o, float* hT, void* ctx, void* stream) {
  if (p && !(p->flags & KDA_FLAG_CHANNEL_GATES))
    return fail(KDA_ERR_INVALID_ARG, "kda_gdn2_fwd needs KDA_FLAG_CHANNEL_GATES in the problem's flags");
  if (p && p->total_tokens > 0) {
    CHECK_PTR(erase_raw);
    CHECK_PTR(write_raw);
  }
  return forward(p, q, k, v, g_raw, erase_raw, write_raw, A_log, dt_bias, h0, o, hT, ctx, stream);
}

kda_status kda_gdn2_bwd(const kda_problem* p, const void* q, const void* k, const void* v, const void* g_raw,
                        const void* erase_raw, const void* write_raw, const float* A_log, const float* dt_bias,
                        const void* dO, const float* dhT, const void* ctx, void* dq, void* dk, void* dv,
                        void* dg_raw, void* derase_raw, void* dwrite_raw, float* dA_log, float* ddt_bias,
                        float* dh0, void* workspace, void* stream) {
  if (p && !(p->flags & KDA_FLAG_CHANNEL_GATES))
    return fail(KDA_ERR_INVALID_ARG, "kda_gdn2_bwd needs KDA_FLAG_CHANNEL_GATES in the problem's flags");
  if (p && p->total_tokens > 0) {
    CHECK_PTR(erase_raw);
    CHECK_PTR(write_raw);
    CHECK_PTR(derase_raw);
    CHECK_PTR(dwrite_raw);
  }
  return backward(p, q, k, v, g_raw, erase_raw, write_raw, A_log, dt_bias, dO, dhT, ctx, dq, dk, dv, dg_raw,
                  derase_raw, dwrite_raw, dA_log, ddt_bias, dh0, workspace, stream);
}

kda_status kda_query_device_status(const void* buf, void* stream) {
  if (!buf) return fail(KDA_ERR_INVALID_ARG, "buffer is NULL");
  cudaStream_t s = (cudaStream_t)stream;
  int word = 0;
  if (cudaMemcpyAsync(&word, buf, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return fail(KDA_ERR_CUDA, "status read failed: %s", cudaGetErrorString(cudaGetLastError()));
  if (word == 0) return KDA_OK;
  if (word == KDA_ERR_TIMEOUT) return fail(KDA_ERR_TIMEOUT, "a device-side bounded wait ran out");
  return fail(KDA_ERR_DEVICE_CHECK, "device-side check failed (code %d)", word);
}

}  // extern "C"
