// kda_noalloc.cu -- kda_bwd_noalloc: the backward for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the
// backward: a host that hands out all device memory from its own fixed pool
// (so a foreign allocation fails or fragments it), a plug-in that is given
// device pointers but no allocator, or a loop that must not take the
// implicit synchronisation an allocation can cause. kda_bwd needs a caller
// workspace; this entry point instead keeps the backward's scratch (the
// gate-parameter partial sums and the recomputed chunk-start states) in one
// fixed-size array that lives inside the library.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds KDA_NOALLOC_SCRATCH_BYTES of it until the process exits. In
// host code the array's name is only a host-side stand-in, never a device
// address, so its device address is looked up once per device with
// cudaGetSymbolAddress (on the first call made with that device current) and
// passed to the kernels. Every call shares the array and it keeps the last
// call's contents; the only word that must start at zero (the status word)
// is cleared on the caller's stream at the start of each call. Two calls
// whose GPU work overlaps (different streams, or different host threads on
// the same device) race on the array and give wrong results: serialise them.
#include <mutex>

#include "kda_internal.cuh"

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
kda_status scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kda::set_error(KDA_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return kda::set_error(KDA_ERR_UNSUPPORTED, "device ordinal %d is beyond the supported %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_kda_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return kda::set_error(KDA_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed: %s",
                            cudaGetErrorString(e));
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" kda_status kda_bwd_noalloc(const kda_problem* p, const void* q, const void* k, const void* v,
                                      const void* g_raw, const void* beta_raw, const float* A_log,
                                      const float* dt_bias, const void* dO, const float* dhT, const void* ctx,
                                      void* dq, void* dk, void* dv, void* dg_raw, void* dbeta_raw,
                                      float* dA_log, float* ddt_bias, float* dh0, void* stream) {
  kda_status st = kda::validate_problem(p);
  if (st != KDA_OK) return st;
  if ((dhT && !aligned16(dhT)) || (dh0 && !aligned16(dh0)))
    return kda::set_error(KDA_ERR_INVALID_ARG, "dhT / dh0 is not 16-byte aligned");
  if (p->flags & KDA_FLAG_CHANNEL_GATES)
    return kda::set_error(KDA_ERR_INVALID_ARG, "KDA_FLAG_CHANNEL_GATES: kda_bwd_noalloc runs KDA only");
  if (p->flags & KDA_FLAG_NO_CHECKPOINTS)
    return kda::set_error(KDA_ERR_INVALID_ARG,
                          "KDA_FLAG_NO_CHECKPOINTS: a forward without checkpoints cannot feed the backward");
  const void* ptrs[] = {q, k, v, g_raw, beta_raw, A_log, dt_bias, dO, ctx, dq, dk, dv, dg_raw, dbeta_raw,
                        dA_log, ddt_bias};
  const char* names[] = {"q", "k", "v", "g_raw", "beta_raw", "A_log", "dt_bias", "dO", "ctx", "dq", "dk", "dv",
                         "dg_raw", "dbeta_raw", "dA_log", "ddt_bias"};
  for (int i = 0; i < 16; ++i) {
    if (ptrs[i] == nullptr) return kda::set_error(KDA_ERR_INVALID_ARG, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return kda::set_error(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  }
  // Scratch plan inside the fixed array: status header, per-(sequence, head)
  // gate-parameter partials, (tensor-core family) the per-item edge tiles,
  // then as many per-CTA state slots as fit.
  // Same kernel family as kda_bwd, so both entry points give identical results.
  const bool tc = kda::kernel_family(p) == 1;
  const size_t edge = tc ? kda::bwd_edge_bytes_tc((int64_t)p->num_seqs * p->num_heads) : 0;
  const size_t head = (size_t)kda::kHeaderBytes + kda::cu_copy_bytes(p->num_seqs) + kda::gate_partial_bytes(p) + edge;
  const size_t per_cta = tc ? kda::bwd_scratch_bytes_per_cta_tc() : kda::bwd_scratch_bytes_per_cta_simt(p);
  const size_t cap = (size_t)KDA_NOALLOC_SCRATCH_BYTES;
  if (head + per_cta > cap)
    return kda::set_error(KDA_ERR_WORKSPACE,
                          "kda_bwd_noalloc needs %zu bytes of scratch for this problem (at least %zu), but its "
                          "fixed buffer holds %zu bytes; use kda_bwd with a caller workspace",
                          head + per_cta, head + per_cta, cap);
  cudaStream_t s = (cudaStream_t)stream;
  if (p->total_tokens == 0) {
    if (cudaMemsetAsync(dA_log, 0, sizeof(float) * p->num_heads, s) != cudaSuccess ||
        cudaMemsetAsync(ddt_bias, 0, sizeof(float) * p->num_heads * p->head_dim, s) != cudaSuccess)
      return kda::set_error(KDA_ERR_CUDA, "memset failed: %s", cudaGetErrorString(cudaGetLastError()));
    if (dh0) {  // no tokens: dh0 = dhT
      const size_t sb = (size_t)p->num_seqs * p->num_heads * p->head_dim * p->head_dim * sizeof(float);
      const cudaError_t e = dhT ? cudaMemcpyAsync(dh0, dhT, sb, cudaMemcpyDeviceToDevice, s)
                                : cudaMemsetAsync(dh0, 0, sb, s);
      if (e != cudaSuccess)
        return kda::set_error(KDA_ERR_CUDA, "state copy failed: %s", cudaGetErrorString(cudaGetLastError()));
    }
    return KDA_OK;
  }
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != KDA_OK) return st;

  const long long items = (long long)p->num_seqs * p->num_heads;
  long long ctas = (long long)((cap - head) / per_cta);
  if (ctas > items) ctas = items;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms > 0 && ctas > sms) ctas = sms;

  kda::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g_raw; a.b = beta_raw; a.A_log = A_log; a.dt_bias = dt_bias;
  a.dO = dO;
  a.dhT = dhT;
  a.dh0 = dh0;
  a.ckpt = (const float*)((const char*)ctx + kda::kHeaderBytes + kda::cu_copy_bytes(p->num_seqs));
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg_raw; a.db = dbeta_raw;
  a.dA_log = dA_log; a.ddt_bias = ddt_bias;
  a.status = (int*)scratch;
  char* ws = (char*)scratch + kda::kHeaderBytes;  // checked copy of cu_seqlens, then the rest
  a.partial = (float*)(ws + kda::cu_copy_bytes(p->num_seqs));
  a.edge = ws + kda::cu_copy_bytes(p->num_seqs) + kda::gate_partial_bytes(p);
  a.scratch = (float*)((char*)scratch + head);
  a.flags = nullptr;  // no helper CTAs here: few CTAs fit the fixed buffer
  a.cu = (const int32_t*)ws;
  a.S = p->total_tokens; a.N = p->num_seqs; a.H = p->num_heads;
  a.scale = p->scale; a.lower = p->gate_lower_bound; a.eps = p->l2_eps;
  if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess)
    return kda::set_error(KDA_ERR_CUDA, "status reset failed: %s", cudaGetErrorString(cudaGetLastError()));
  if (kda::launch_check_cu(p->cu_seqlens, p->num_seqs, p->total_tokens, (int32_t*)ws, a.status, s) != KDA_OK)
    return kda::set_error(KDA_ERR_CUDA, "cu_seqlens check launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  st = tc ? kda::launch_bwd_tc(p, a, s, (int)ctas) : kda::launch_bwd_simt_ctas(p, a, s, (int)ctas);
  if (st != KDA_OK)
    return kda::set_error(st, "no-alloc backward launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  return KDA_OK;
}

// The status word of the last kda_bwd_noalloc call on the current device: it
// sits at the head of the library's scratch array, so it is read here with a
// copy from the symbol into a host int (no allocation). Synchronises `stream`.
extern "C" kda_status kda_noalloc_device_status(void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  int word = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&word, g_kda_noalloc_scratch, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return kda::set_error(KDA_ERR_CUDA, "no-alloc status read failed: %s", cudaGetErrorString(e));
  if (word == 0) return KDA_OK;
  if (word == KDA_ERR_TIMEOUT) return kda::set_error(KDA_ERR_TIMEOUT, "a device-side bounded wait ran out");
  return kda::set_error(KDA_ERR_DEVICE_CHECK, "device-side check failed (code %d)", word);
}
