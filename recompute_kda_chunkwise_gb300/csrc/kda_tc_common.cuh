// kda_tc_common.cuh -- inline-PTX helpers for the sm_103a tensor-core (tcgen05)
// KDA kernels: TMEM allocation, tcgen05.mma issue/commit, TMEM loads, TMA
// tensor-tile loads, mbarriers (every wait bounded) and the shared-memory
// matrix layout the MMAs read.
//
// Operand layout used everywhere ("SW128 tile"): a bf16 matrix of R rows x K
// columns (K a multiple of 64) stored K-major with the 128-byte swizzle: the
// K extent is cut into 64-element blocks of R x 128 bytes each; inside a
// block, row r occupies bytes (r/8)*1024 + (r%8)*128, and its 16-byte chunk c
// (elements 8c..8c+7) is stored at chunk position c ^ (r%8). This is also
// exactly what a TMA tile load with 128-byte swizzle writes for a 64-element
// wide box. The same bytes read "MN-major" describe a K x R operand whose R
// (M or N) extent is contiguous; the MMA descriptor then takes the stride
// between 64-element R blocks as its leading byte offset.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "kda_internal.cuh"

// Stage timers, for a tracing build only (compiled with -DKDA_STAGE_TIMERS).
// Thread 0 of each CTA adds the clock64 cycles since its previous mark to a
// per-stage counter in KDA_STAGE_BYTES of shared memory (slot 31 counts the
// steps); the counters go to the CTA's row of a device array when the CTA
// exits. In the default build every mark compiles to nothing and no shared
// memory is set aside.
#ifdef KDA_STAGE_TIMERS
#define KDA_STAGE_BYTES 128
#define KDA_STAGE_INIT(smem_ptr)                                            \
  unsigned* const kda_stage_sm = reinterpret_cast<unsigned*>(smem_ptr);     \
  long long kda_stage_t = clock64();                                        \
  if (threadIdx.x == 0)                                                     \
    for (int i_ = 0; i_ < 32; ++i_) kda_stage_sm[i_] = 0u
#define KDA_STAGE(id)                                                       \
  do {                                                                      \
    if (threadIdx.x == 0) {                                                 \
      const long long t_ = clock64();                                       \
      kda_stage_sm[(id)] += static_cast<unsigned>(t_ - kda_stage_t);        \
      kda_stage_t = t_;                                                     \
    }                                                                       \
  } while (0)
#define KDA_STAGE_STEP()                                                    \
  do {                                                                      \
    if (threadIdx.x == 0) kda_stage_sm[31] += 1u;                           \
  } while (0)
#define KDA_STAGE_FLUSH(dev_array)                                          \
  do {                                                                      \
    if (threadIdx.x == 0 && blockIdx.x < kStageCtas)                        \
      for (int i_ = 0; i_ < 32; ++i_) (dev_array)[blockIdx.x * 32 + i_] += kda_stage_sm[i_]; \
  } while (0)
#else
#define KDA_STAGE_BYTES 0
#define KDA_STAGE_INIT(smem_ptr) \
  do {                           \
  } while (0)
#define KDA_STAGE(id) \
  do {                \
  } while (0)
#define KDA_STAGE_STEP() \
  do {                   \
  } while (0)
#define KDA_STAGE_FLUSH(dev_array) \
  do {                             \
  } while (0)
#endif
// CTAs whose stage counters a tracing build keeps (rows of its device array)
constexpr int kStageCtas = 512;

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (row, k) inside an SW128 tile of `rows` rows.
__device__ __forceinline__ uint32_t sw128_off(int row, int k, int rows) {
  const int kb = k >> 6, w = k & 63, chunk = w >> 3, e = w & 7;
  return static_cast<uint32_t>(kb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                               ((chunk ^ (row & 7)) << 4) + (e << 1));
}
// Byte offset of the 16-byte chunk holding elements (row, 8c .. 8c+7).
__device__ __forceinline__ uint32_t sw128_chunk(int row, int c, int rows) {
  const int kb = c >> 3, ch = c & 7;
  return static_cast<uint32_t>(kb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4));
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// byte offset, stride byte offset (8-row groups, 1024 B here), version 1,
// layout type 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// K-major operand: K-step ks (16 elements) of the rows [row0, row0 + n) of an
// SW128 tile with `rows` rows at shared address `tile`.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int rows, int row0, int ks) {
  return sdesc(tile + (ks >> 2) * rows * 128 + (row0 >> 3) * 1024 + (ks & 3) * 32, 16);
}
// MN-major operand stored as an SW128 tile whose rows are the K index and
// whose 64-element column blocks (stride `block_bytes`) run along M/N.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int block_bytes, int ks) {
  return sdesc(tile + ks * 2048, block_bytes);
}

// The same descriptors as offsets from a base descriptor D0 = sdesc(smem
// base, 0) of a 1024-byte aligned shared-memory base: the start field
// (address / 16, 14 bits) and the leading-byte-offset field are plain sums
// that never carry, so with a constant `off` each descriptor is D0 plus a
// compile-time constant (one add at issue time).
__device__ __forceinline__ uint64_t desc_k(uint64_t D0, uint32_t off, int rows, int row0, int ks) {
  return D0 + ((static_cast<uint64_t>((off + (ks >> 2) * rows * 128 + (row0 >> 3) * 1024 + (ks & 3) * 32) >> 4)) |
               (static_cast<uint64_t>(16 >> 4) << 16));
}
__device__ __forceinline__ uint64_t desc_mn(uint64_t D0, uint32_t off, int block_bytes, int ks) {
  return D0 + ((static_cast<uint64_t>((off + ks * 2048) >> 4)) | (static_cast<uint64_t>(block_bytes >> 4) << 16));
}

// Instruction descriptors (fp32 accumulate, shape M x N, optional MN-major
// A / B): kind::f16 with fp16 A and B (format 0), kind::tf32 (format 2).
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn = false, bool b_mn = false) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D (+)= A B with A and B in shared memory (kind::f16, fp16 operands).
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
// D (+)= A B, kind::tf32, A read from TMEM (lane = row, one 32-bit column per
// K element), B from shared memory.
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes -> visible to tcgen05 / TMA (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit values: thread (lane) gets 32 consecutive
// columns of TMEM lane (warp's lane quarter base + lane).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 8 columns of the thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}

// Stores 32 consecutive 32-bit columns of the thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31]));
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
// Bounded wait for the phase with the given parity to complete. Returns
// false (and records KDA_ERR_TIMEOUT) if it did not complete within `limit`
// polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, int limit = 1 << 24) {
  const uint32_t a = smem_addr(bar);
  for (int it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  set_status(status, KDA_ERR_TIMEOUT);
  return false;
}

// TMA: 3-D tile (x = channel, y = head, z = token) of a [S][H][D] tensor into
// shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of element (row, k) in a 32-bit SW128 tile of `rows` rows (the
// K extent cut into 32-element blocks of rows x 128 bytes).
__device__ __forceinline__ uint32_t sw128_off32(int row, int k, int rows) {
  const int kb = k >> 5, w = k & 31, chunk = w >> 2, e = w & 3;
  return static_cast<uint32_t>(kb * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                               ((chunk ^ (row & 7)) << 4) + (e << 2));
}

// ---- per-thread async copies (16 bytes; src_bytes = 0 writes zeros) ----
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most the newest group of this thread's copies is pending.
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// ---- bulk (non-tensor) async copies between shared and global memory ----
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The source shared memory of every committed bulk store may be reused.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The source shared memory of all but the N most recent bulk stores may be reused.
template <int N>
__device__ __forceinline__ void bulk_wait_read_but() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Every committed bulk store has completed (its writes are visible).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---- warp-level tf32 tensor-core tiles (mma.sync m16n8k8) for 16-row work ----
// Fragment layout (g = lane / 4, t = lane % 4): A[16 x 8] rows g, g + 8 and
// columns t, t + 4 in a0..a3 = (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4);
// B[8 x 8] b0 = (k = t, n = g), b1 = (k = t + 4, n = g); C[16 x 8]
// c0..c3 = (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  lo = __float_as_uint(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32_16x8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// d += A B with both operands split into tf32 hi + lo parts (hi*hi + hi*lo +
// lo*hi): about fp32 accuracy.
__device__ __forceinline__ void mma3(float (&d)[4], const float (&a)[4], const float (&b)[2]) {
  uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
  split_tf32(b[0], bh[0], bl[0]);
  split_tf32(b[1], bh[1], bl[1]);
  mma_tf32_16x8(d, al[0], al[1], al[2], al[3], bh[0], bh[1]);
  mma_tf32_16x8(d, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
  mma_tf32_16x8(d, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
}
// d += A B in plain tf32 (both operands rounded to tf32 once): about 2^-11
// relative per product, for results that feed nothing more sensitive.
__device__ __forceinline__ void mma1(float (&d)[4], const float (&a)[4], const float (&b)[2]) {
  uint32_t ah[4], bh[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(ah[i]) : "f"(a[i]));
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(bh[0]) : "f"(b[0]));
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(bh[1]) : "f"(b[1]));
  mma_tf32_16x8(d, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
}
// d += A B where B is exact in tf32 (bf16 / fp16 values): A split only.
__device__ __forceinline__ void mma2_bexact(float (&d)[4], const float (&a)[4], const float (&b)[2]) {
  uint32_t ah[4], al[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
  const uint32_t b0 = __float_as_uint(b[0]), b1 = __float_as_uint(b[1]);
  mma_tf32_16x8(d, al[0], al[1], al[2], al[3], b0, b1);
  mma_tf32_16x8(d, ah[0], ah[1], ah[2], ah[3], b0, b1);
}
// d += A B where A is exact in tf32: B split only.
__device__ __forceinline__ void mma2_aexact(float (&d)[4], const float (&a)[4], const float (&b)[2]) {
  uint32_t bh[2], bl[2];
  split_tf32(b[0], bh[0], bl[0]);
  split_tf32(b[1], bh[1], bl[1]);
  const uint32_t a0 = __float_as_uint(a[0]), a1 = __float_as_uint(a[1]), a2 = __float_as_uint(a[2]),
                 a3 = __float_as_uint(a[3]);
  mma_tf32_16x8(d, a0, a1, a2, a3, bl[0], bl[1]);
  mma_tf32_16x8(d, a0, a1, a2, a3, bh[0], bh[1]);
}

// mma.sync fragment loads from fp32 row-major shared-memory matrices (g = lane / 4,
// t = lane % 4; ld = row stride in floats)
// A[m][k] = X[m][k]
__device__ __forceinline__ void ldA(float (&a)[4], const float* X, int ld, int k0, int g, int t) {
  a[0] = X[g * ld + k0 + t];
  a[1] = X[(g + 8) * ld + k0 + t];
  a[2] = X[g * ld + k0 + t + 4];
  a[3] = X[(g + 8) * ld + k0 + t + 4];
}
// A[m][k] = X[k][m]
__device__ __forceinline__ void ldAT(float (&a)[4], const float* X, int ld, int k0, int g, int t) {
  a[0] = X[(k0 + t) * ld + g];
  a[1] = X[(k0 + t) * ld + g + 8];
  a[2] = X[(k0 + t + 4) * ld + g];
  a[3] = X[(k0 + t + 4) * ld + g + 8];
}
// B[k][n] = Y[n][k]
__device__ __forceinline__ void ldBc(float (&b)[2], const float* Y, int ld, int n0, int k0, int g, int t) {
  b[0] = Y[(n0 + g) * ld + k0 + t];
  b[1] = Y[(n0 + g) * ld + k0 + t + 4];
}
// B[k][n] = Z[k][n]
__device__ __forceinline__ void ldBr(float (&b)[2], const float* Z, int ld, int n0, int k0, int g, int t) {
  b[0] = Z[(k0 + t) * ld + n0 + g];
  b[1] = Z[(k0 + t + 4) * ld + n0 + g];
}

// ---- cross-CTA hand-off between co-resident CTAs of one cooperative launch
// (every wait bounded) ----
__device__ __forceinline__ bool wait_flag_geq(const uint32_t* f, uint32_t target, int* status) {
  for (int it = 0; it < (1 << 24); ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v >= target) return true;
    __nanosleep(64);
  }
  set_status(status, KDA_ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ void st_release(uint32_t* f, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
// barrier `id` (1..15) over the first `n` threads of the CTA (n a multiple of 32)
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// orders this thread's generic-proxy accesses with its async-proxy accesses of global memory
__device__ __forceinline__ void fence_proxy_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Raw bits of one bf16 element (the caller converts where it uses the value,
// so that nothing waits on the load before then).
__device__ __forceinline__ unsigned short beta_bits(const __nv_bfloat16* p, int64_t i) {
  return reinterpret_cast<const unsigned short*>(p)[i];
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 p = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(p);
}

}  // namespace tc
}  // namespace kda
