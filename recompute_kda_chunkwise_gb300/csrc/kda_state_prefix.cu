// kda_state_prefix.cu -- the affine state prefix that joins the pieces of a
// sequence cut in time (context parallelism).
//
// The recurrence is linear in its state: for fixed inputs, a piece of a
// sequence maps the state it starts from to the state it ends with through
// an affine map, H_end = A H_start + B, where A (D x D, acting on the key
// index) is the piece run from the identity with zero values and B the piece
// run from zero with its values. The backward is the transposed map: the
// gradient at the piece's start is A^T (gradient at its end) + C, where C is
// the start-state gradient of the piece's own backward run from a zero
// end-state gradient. Once every piece's map is known, a short prefix over
// the pieces gives each piece its true start state (forward) or its true
// end-state gradient (backward), and the pieces then run independently.
// This is the exchange step of the context-parallel split (the page "KDA
// Memory with Recompute ...", section "Measured peak allocated memory",
// leaves every 256K-token case unmeasured: the lengths that call for it);
// on several GPUs the maps are gathered from the ranks first, on one GPU the
// pieces are packed sequences of one launch.
//
// One CTA per (sequence, head): P dependent D x D x D products in fp32,
// with the running state and the piece's matrix staged in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kPT = 256;

// Row stride of the staged matrix (padded: threads of a warp read one column
// of it at once).
template <int D>
struct PrefixSmem {
  static constexpr int LDM = D + 1;
  static constexpr size_t bytes = static_cast<size_t>(D) * LDM * 4 + static_cast<size_t>(D) * D * 4;
};

// direction 0: x_{p+1} = A_p x_p + B_p, x_0 = x0, xs[p] = x_p, x_end = x_P.
// direction 1: x_{p-1} = A_p^T x_p + B_p, x_{P-1} = x0, xs[p] = x_p, x_end = A_0^T x_0 + B_0.
// CTA (n, h) = (blockIdx.x / H, blockIdx.x % H); its matrix for piece p sits
// at (p * piece_stride + n * seq_stride + h) * D * D in A, B and xs, and at
// (n * H + h) * D * D in x0 and x_end.
template <int D>
__global__ void __launch_bounds__(kPT) kda_state_prefix_kernel(int pieces, int H, int direction,
                                                               int64_t piece_stride, int64_t seq_stride,
                                                               const float* __restrict__ A,
                                                               const float* __restrict__ B,
                                                               const float* __restrict__ x0, float* xs,
                                                               float* x_end) {
  constexpr int LDM = PrefixSmem<D>::LDM;
  constexpr int TPR = kPT / D;     // threads per output row
  constexpr int CPT = D / TPR;     // output columns per thread
  extern __shared__ float psm[];
  float* M = psm;                  // [D][LDM] the piece's matrix (A or A^T)
  float* X = psm + D * LDM;        // [D][D]   the running state
  const int item = blockIdx.x, tid = threadIdx.x;
  const int n = item / H, h = item % H;
  const int row = tid / TPR, col0 = (tid % TPR) * CPT;
  const int64_t mat = static_cast<int64_t>(D) * D;
  const float* src0 = x0 ? x0 + item * mat : nullptr;
  for (int x = tid; x < D * D; x += kPT) X[x] = src0 ? src0[x] : 0.f;
  for (int step = 0; step < pieces; ++step) {
    const int p = direction == 0 ? step : pieces - 1 - step;
    const int64_t off = (p * piece_stride + n * seq_stride + h) * mat;
    // the state entering this step is piece p's start state (forward) or
    // its end-state gradient (backward)
    __syncthreads();
    for (int x = tid; x < D * D; x += kPT) xs[off + x] = X[x];
    const float* Ap = A + off;
    if (direction == 0) {
      for (int x = tid; x < D * D; x += kPT) M[(x / D) * LDM + x % D] = Ap[x];
    } else {
      for (int x = tid; x < D * D; x += kPT) M[(x % D) * LDM + x / D] = Ap[x];  // A^T
    }
    __syncthreads();
    float acc[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) acc[j] = B[off + static_cast<int64_t>(row) * D + col0 + j];
    for (int k = 0; k < D; ++k) {
      const float m = M[row * LDM + k];
#pragma unroll
      for (int j = 0; j < CPT; ++j) acc[j] = fmaf(m, X[k * D + col0 + j], acc[j]);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < CPT; ++j) X[row * D + col0 + j] = acc[j];
  }
  __syncthreads();
  if (x_end != nullptr)
    for (int x = tid; x < D * D; x += kPT) x_end[item * mat + x] = X[x];
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_state_prefix(int32_t num_seqs, int32_t pieces, int32_t num_heads, int32_t head_dim,
                                       int32_t direction, int64_t piece_stride, int64_t seq_stride,
                                       const float* A, const float* B, const float* x0, float* xs, float* x_end,
                                       void* stream) {
  if (num_seqs < 0 || pieces < 1 || num_heads < 1)
    return kda::set_error(KDA_ERR_INVALID_ARG, "need num_seqs >= 0, pieces >= 1, num_heads >= 1");
  if (head_dim != 64 && head_dim != 128)
    return kda::set_error(KDA_ERR_UNSUPPORTED, "head_dim %d is not supported (64 or 128)", head_dim);
  if (direction != KDA_PREFIX_FORWARD && direction != KDA_PREFIX_BACKWARD)
    return kda::set_error(KDA_ERR_INVALID_ARG, "direction must be KDA_PREFIX_FORWARD or KDA_PREFIX_BACKWARD");
  // the matrix offsets (p * piece_stride + n * seq_stride + h) must be distinct and non-negative
  if (piece_stride < 0 || seq_stride < 0 ||
      !((piece_stride >= num_heads && seq_stride >= (int64_t)pieces * piece_stride) ||
        (seq_stride >= num_heads && piece_stride >= (int64_t)num_seqs * seq_stride)))
    return kda::set_error(KDA_ERR_INVALID_ARG, "piece_stride / seq_stride do not describe a [pieces][seqs][heads] "
                          "or [seqs][pieces][heads] layout");
  if ((int64_t)num_seqs * num_heads > (1 << 30)) return kda::set_error(KDA_ERR_INVALID_ARG, "too many sequences x heads");
  if (num_seqs == 0) return KDA_OK;
  if (!A || !B || !xs) return kda::set_error(KDA_ERR_INVALID_ARG, "A, B and xs must not be NULL");
  const void* ptrs[] = {A, B, x0, xs, x_end};
  for (const void* q : ptrs)
    if (q && ((uintptr_t)q & 15u)) return kda::set_error(KDA_ERR_INVALID_ARG, "state buffers must be 16-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  const int dir = direction == KDA_PREFIX_FORWARD ? 0 : 1;
  const int grid = num_seqs * num_heads;
  if (head_dim == 128) {
    constexpr size_t smem = kda::PrefixSmem<128>::bytes;
    if (cudaFuncSetAttribute(kda::kda_state_prefix_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return kda::set_error(KDA_ERR_CUDA, "prefix kernel attribute: %s", cudaGetErrorString(cudaGetLastError()));
    kda::kda_state_prefix_kernel<128><<<grid, kda::kPT, smem, s>>>(pieces, num_heads, dir, piece_stride, seq_stride,
                                                                   A, B, x0, xs, x_end);
  } else {
    constexpr size_t smem = kda::PrefixSmem<64>::bytes;
    kda::kda_state_prefix_kernel<64><<<grid, kda::kPT, smem, s>>>(pieces, num_heads, dir, piece_stride, seq_stride,
                                                                  A, B, x0, xs, x_end);
  }
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? KDA_OK : kda::set_error(KDA_ERR_CUDA, "prefix launch failed: %s", cudaGetErrorString(e));
}
