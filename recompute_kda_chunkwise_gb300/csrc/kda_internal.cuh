// kda_internal.cuh -- constants, argument blocks and small device helpers
// shared by the KDA kernels. Not part of the public ABI (include/kda.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Tokens between two state checkpoints stored by the forward in ctx (one
// fp32 D x D state per checkpoint, sequence and head).
constexpr int kCkptTokens = 1024;
// Bytes reserved at the head of ctx / workspace for the device status word.
constexpr int kHeaderBytes = 256;
// Upper bound on backward CTAs (persistent grid), which sizes the workspace.
constexpr int kMaxBwdCtas = 304;

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  void* o;
  const float* h0;  // initial states [N][H][D][D] (NULL: zero)
  float* hT;        // final states (NULL: not written)
  float* ckpt;  // NULL: no checkpoints
  int* status;  // NULL when ckpt is NULL
  const int32_t* cu;
  int64_t S;  // total tokens (cu[N])
  int N, H;
  float scale, lower, eps;
  int test_timeout;  // KDA_FLAG_TEST_TIMEOUT (tensor-core forward only)
  // tensor-core forward, split mode: per-item hand-off counters and slots in
  // ctx (NULL: no helper CTAs)
  uint32_t* xflags;
  uint8_t* xbuf;
  // GDN-2 (KDA_FLAG_CHANNEL_GATES): raw write gate [S,H,D]; b is then the
  // raw erase gate [S,H,D]
  const void* w = nullptr;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* b;
  const float* A_log;
  const float* dt_bias;
  const void* dO;
  const float* dhT;  // gradient of the final states [N][H][D][D] (NULL: zero)
  float* dh0;        // gradient of the initial states (NULL: not written)
  const float* ckpt;
  void* dq;
  void* dk;
  void* dv;
  void* dg;
  void* db;
  float* dA_log;
  float* ddt_bias;
  float* partial;  // [N*H][D+1]
  float* scratch;  // per-CTA segment states
  void* edge = nullptr;  // tensor-core backward: per-item low parts of the sequence-edge chunk states
  uint32_t* flags;  // tensor-core backward: per-item hand-off counters (NULL: no helper CTAs)
  int* status;
  const int32_t* cu;
  int64_t S;  // total tokens (cu[N])
  int N, H;
  float scale, lower, eps;
  // GDN-2 (KDA_FLAG_CHANNEL_GATES, CUDA-core backward only): raw write gate
  // and its gradient [S,H,D]; b / db are then the raw erase gate and its
  // gradient [S,H,D]
  const void* w = nullptr;
  void* dw = nullptr;
};

// Index of the checkpoint slot of (sequence n, segment j) relative to slot 0:
// floor(cu[n] / kCkptTokens) + n + j. Sequence n owns ceil(T_n / kCkptTokens)
// consecutive slots and these ranges never overlap, so the total count is
// bounded by floor(S / kCkptTokens) + N (see kda_ctx_bytes).
__host__ __device__ inline int64_t ckpt_slot(int64_t bos, int n, int j) {
  return bos / kCkptTokens + n + j;
}

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }
// sigmoid'(x) = sigmoid(x) sigmoid(-x): both factors are computed directly,
// so the result keeps its relative accuracy where sigmoid(x) is near 1
// (1 - sigmoid(x) would cancel there).
__device__ __forceinline__ float sigmoid_grad(float x) { return sigmoidf_(x) * sigmoidf_(-x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}


// Host-side launchers (defined in the kernel translation units).
kda_status launch_fwd_simt(const kda_problem* p, const FwdArgs& a, cudaStream_t s);
kda_status launch_fwd_tc(const kda_problem* p, const FwdArgs& a, cudaStream_t s);
// the forward with 16-token chunks (KDA_FLAG_CHUNK16), on the backward kernel's stages
kda_status launch_fwd16_tc(const kda_problem* p, const FwdArgs& a, cudaStream_t s);
kda_status launch_bwd_simt(const kda_problem* p, const BwdArgs& a, cudaStream_t s);
size_t bwd_scratch_bytes_simt(const kda_problem* p, int* nctas);
kda_status launch_bwd_simt_ctas(const kda_problem* p, const BwdArgs& a, cudaStream_t s, int ctas);
size_t bwd_scratch_bytes_per_cta_simt(const kda_problem* p);
size_t bwd_scratch_bytes_per_cta_tc();
size_t bwd_scratch_bytes_per_buf_split_tc();
// Bytes of the tensor-core backward's per-item edge area (low parts of the
// first and last chunk's start states).
size_t bwd_edge_bytes_tc(int64_t items);
// Bytes of the tensor-core forward's hand-off area (counters + slots) for
// `items` (sequence, head) items.
size_t fwd_handoff_bytes(int items);
kda_status launch_bwd_tc(const kda_problem* p, const BwdArgs& a, cudaStream_t s, int ctas);
// CTAs of the tensor-core backward: one per SM of a 152-SM part (persistent).
constexpr int kTcBwdCtas = 152;
// Split-mode backward: segment buffers per item (helpers rebuild up to
// kTcBwdBufs - 1 levels ahead of the reverse CTA) and hand-off counters per
// item (one "rebuilt" counter per buffer, then one "consumed" counter).
constexpr int kTcBwdBufs = 3;
constexpr int kTcBwdFlags = kTcBwdBufs + 1;

// Bytes of the checked copy of cu_seqlens that follows the header of ctx
// and workspace (and of the no-allocation scratch array).
inline size_t cu_copy_bytes(int num_seqs) { return ((size_t)(num_seqs + 1) * sizeof(int32_t) + 255) / 256 * 256; }
// Enqueues the device-side check of cu_seqlens: cu_out = cu when cu[0] == 0,
// cu is non-decreasing and cu[N] == S; otherwise cu_out = all zeros (every
// sequence empty) and KDA_ERR_DEVICE_CHECK in *status. The kernels then read
// cu_out only.
kda_status launch_check_cu(const int32_t* cu, int N, int64_t S, int32_t* cu_out, int* status, cudaStream_t s);

// Host helpers shared by the entry points (defined in kda_api.cu).
kda_status validate_problem(const kda_problem* p);
kda_status set_error(kda_status s, const char* fmt, ...);
size_t gate_partial_bytes(const kda_problem* p);
// 1: tcgen05 kernels (bf16, head_dim 128, no KDA_FLAG_FORCE_SIMT), else 0: fp32 SIMT kernels.
int kernel_family(const kda_problem* p);

}  // namespace kda
