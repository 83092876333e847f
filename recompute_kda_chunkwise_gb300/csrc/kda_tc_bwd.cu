// kda_tc_bwd.cu -- tensor-core KDA backward (bf16 inputs, D = K = V = 128) with
// the recompute policy: the forward keeps one fp32 state per 1024 tokens; per
// such segment (walked in reverse) the backward rebuilds the chunk-start
// states, keeps them as fp16 tiles in per-CTA scratch, then walks the
// segment's chunks in reverse, recomputing each chunk's WY factors and gated
// q/k from the inputs and propagating the state gradient dH.
//
// Chunk size C = 16: every factor exp(+-(G_r - G_s)) inside a chunk then stays
// within fp32 range (the "k/exp(cumsum g) underflows past 17 tokens" note of
// "KDA at the production shape ...", section 3(a)), so the intra-chunk
// matrices and all their gradients are plain fp32 products on CUDA cores,
// while every product with a 128-long contraction or a 128 x 128 result
// (the state terms) runs on tcgen05 with fp16 operands and fp32 accumulators
// in TMEM (M = 128 with the value index v or the key index i on the lanes).
// Both fp32 states live in TMEM (H^T during the rebuild, dH^T throughout).
//
// Per chunk (r, s in 0..15; G chunk-local cumulative log-decay; Gamma = e^G;
// T' = T diag(beta), T = (I + diag(beta) Abar)^-1):
//   U~ = T' V - T' (Kh Gamma) H          O-side:  dQG = dO H^T,  dM = dO U~^T
//   dU~ = M^T dO + Kbar dH'               dH = diag(gamma) dH' + (Qh Gamma)^T dO - W^T dU~
//   dW = -dU~ H^T,  dKbar = U~ dH'^T,  dgamma = rowsum(H .* dH')
//   dT' = dW (Kh Gamma)^T + dU~ V^T,  dV = T'^T dU~,  d(Kh Gamma) += T'^T dW
//   dA = -T^T (dT' diag(beta)) T^T,  then Abar / M / gate / L2-norm chain rules.
#include "kda_tc_common.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kC = 16;
constexpr int kD = 128;
constexpr int kT = 256;
constexpr int kCPS = kCkptTokens / kC;  // chunks per checkpoint segment (64)
constexpr int kLd = 132;                // fp32 tile row stride (floats)
constexpr int kTile = kC * kLd;         // floats per fp32 tile
constexpr int kSq = 17;                 // 16 x 16 matrices, row stride
constexpr float kLog2e = 1.4426950408889634f;

// fp32 tiles [16][132]
enum { T_GS = 0, T_QG, T_KG, T_KI, T_KB, T_V, T_DO, T_W, T_U, T_DU, T_AQ, T_AK, T_AG, NT32 };
constexpr int OFF_A1 = 110592;           // H^T fp16 [128 v][128 i] (SW128)
constexpr int OFF_A1D = OFF_A1 + 32768;  // dH'^T fp16 [128 v][128 i]
constexpr int OFF_FW = OFF_A1D + 32768;  // -W     fp16 [16 r][128 i]
constexpr int OFF_FQG = OFF_FW + 4096;   // Qh*Gamma fp16 [16 r][128 i]
constexpr int OFF_FKB = OFF_FQG + 4096;  // Kbar   fp16 [16 r][128 i]
constexpr int OFF_FDO = OFF_FKB + 4096;  // dO     fp16 [16 r][128 v]
constexpr int OFF_FU = OFF_FDO + 4096;   // U~     fp16 [16 r][128 v]
constexpr int OFF_FDU = OFF_FU + 4096;   // dU~    fp16 [16 r][128 v]
constexpr int OFF_FM = OFF_FDU + 4096;   // M hi   fp16 [16 r][64 (16 used) s]
constexpr int OFF_FML = OFF_FM + 2048;   // M lo
constexpr int OFF_SMALL = OFF_FML + 2048;
// small fp32 arrays (offsets in floats)
constexpr int S_AB = 0, S_AQK = 272, S_T = 544, S_TP = 816, S_DM = 1088, S_DTP = 1360, S_DA = 1632, S_Y = 1904;
constexpr int S_BETA = 2176, S_IQ0 = 2192, S_IK0 = 2208, S_DB = 2224, S_RQ = 2240, S_RK = 2256;
constexpr int S_GEND = 2272, S_DGE = 2400, S_TOT = 2528, S_RED = 2784, S_PART = 3296;
constexpr int SMALL_FLOATS = 3584;
constexpr int OFF_BAR = OFF_SMALL + SMALL_FLOATS * 4;
constexpr int SMEM_BYTES = OFF_BAR + 64 + 1024;
static_assert(NT32 * kTile * 4 <= OFF_A1, "fp32 tiles");

// TMEM columns
constexpr uint32_t TM_H = 0;     // H^T fp32 state (rebuild pass), 128
constexpr uint32_t TM_DH = 128;  // dH^T fp32 state, 128
constexpr uint32_t TM_D2 = 256;  // state increment, 128
constexpr uint32_t TM_D1 = 384;  // -(W H)^T [v][r], 16
constexpr uint32_t TM_DU = 400;  // dU~^T [v][r], 16
constexpr uint32_t TM_DQ = 416;  // (H dO^T)[i][r], 16
constexpr uint32_t TM_DW = 432;  // (H dU~^T)[i][r], 16
constexpr uint32_t TM_DK = 448;  // (dH' U~^T)[i][r], 16
constexpr uint32_t TM_COLS = 512;

struct TcBwdArgs {
  const __nv_bfloat16 *q, *k, *v, *g, *b, *dO;
  const float* A_log;
  const float* dt_bias;
  const float* ckpt;
  __nv_bfloat16 *dq, *dk, *dv, *dg, *db;
  float* partial;
  uint4* scratch;  // per CTA: kCPS fp16 state tiles of 32 KB
  int* status;
  const int32_t* cu;
  int N, H;
  float scale, lower, eps;
};

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + ex2(-x * kLog2e)); }
__device__ __forceinline__ void st_h(uint8_t* base, uint32_t off, float x) {
  *reinterpret_cast<__half*>(base + off) = __float2half_rn(x);
}
__device__ __forceinline__ float lo_part(float x) { return x - __half2float(__float2half_rn(x)); }

// Sums 64 per-lane values over the 32 lanes of a warp (recursive halving):
// afterwards lane l holds the totals of indices idx(l, 0) and idx(l, 1) with
// idx(l, e) = 32*b4 + 16*b3 + 8*b2 + 4*b1 + 2*b0 + e (b = bits of l).
__device__ __forceinline__ void warp_reduce_scatter64(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int w = 16 >> step, n = 64 >> step, half = n >> 1;
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < half) {
        const float send = up ? v[j] : v[j + half];
        const float keep = up ? v[j + half] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
  }
}

__global__ void __launch_bounds__(kT, 1) kda_bwd_tc_kernel(const TcBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(sm);
  float* F = reinterpret_cast<float*>(sm);
  float* GS = F + T_GS * kTile;
  float* QG = F + T_QG * kTile;
  float* KG = F + T_KG * kTile;
  float* KI = F + T_KI * kTile;
  float* KB = F + T_KB * kTile;
  float* VT = F + T_V * kTile;
  float* DOT = F + T_DO * kTile;
  float* WT = F + T_W * kTile;
  float* UT = F + T_U * kTile;
  float* DUT = F + T_DU * kTile;
  float* AQ = F + T_AQ * kTile;
  float* AK = F + T_AK * kTile;
  float* AG = F + T_AG * kTile;
  float* S = reinterpret_cast<float*>(sm + OFF_SMALL);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 1);
  int* s_fail = reinterpret_cast<int*>(bar + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ci = tid & 127, rh = tid >> 7;  // channel role: channel ci, rows 8*rh .. 8*rh+7
  const int q4 = warp & 3, hh = warp >> 2, L = 32 * q4 + lane;  // lane role
  const uint32_t tlane = static_cast<uint32_t>(32 * q4) << 16;
  const int sr = tid >> 4, ss = tid & 15;  // (r, s) role for 16 x 16 matrices
  const float Lg = a.lower * kLog2e;

  if (tid == 0) {
    mbar_init(bar, 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(s_tmem, TM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *s_tmem;
  uint32_t ph = 0;
  uint4* scratch = a.scratch + static_cast<size_t>(blockIdx.x) * kCPS * (32768 / 16);

#define KDA_WAIT_MMA()                                  \
  do {                                                  \
    if (!mbar_wait(bar, ph, a.status)) *s_fail = 1;     \
    ph ^= 1u;                                           \
  } while (0)
#define KDA_SYNC_OR_BAIL()      \
  do {                          \
    __syncthreads();            \
    if (*s_fail) goto teardown; \
  } while (0)

  for (int item = blockIdx.x; item < a.N * a.H; item += gridDim.x) {
    const int n = item / a.H, h = item % a.H;
    const int64_t bos = a.cu[n], eos = a.cu[n + 1];
    const int nchunks = static_cast<int>((eos - bos + kC - 1) / kC);
    const int nseg = static_cast<int>((eos - bos + kCkptTokens - 1) / kCkptTokens);
    const float expA = expf(a.A_log[h]);
    const float dtb = a.dt_bias[h * kD + ci];
    float acc_dtb = 0.f, acc_alog = 0.f;

    // dH' = 0 (TMEM state and its fp16 operand copy)
    {
      float z[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = 0.f;
      tmem_st32(tmem + tlane + TM_DH + 64 * hh, z);
      tmem_st32(tmem + tlane + TM_DH + 64 * hh + 32, z);
      tmem_st_wait();
      for (int x = tid; x < 32768 / 16; x += kT) reinterpret_cast<uint4*>(sm + OFF_A1D)[x] = make_uint4(0, 0, 0, 0);
    }

    for (int seg = nseg - 1; seg >= 0; --seg) {
      const int c0 = seg * kCPS, c1 = min(nchunks, c0 + kCPS);
      // ---- segment start state: checkpoint (fp32 [i][v]) -> TMEM H^T and fp16 A1 ----
      {
        const float* src = a.ckpt + (ckpt_slot(bos, n, seg) * a.H + h) * static_cast<int64_t>(kD * kD);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = src[(64 * hh + 32 * half + j) * kD + L];
          tmem_st32(tmem + tlane + TM_H + 64 * hh + 32 * half, x);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            *reinterpret_cast<uint4*>(sm + OFF_A1 + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)) =
                make_uint4(pack_h2(x[8 * cc], x[8 * cc + 1]), pack_h2(x[8 * cc + 2], x[8 * cc + 3]),
                           pack_h2(x[8 * cc + 4], x[8 * cc + 5]), pack_h2(x[8 * cc + 6], x[8 * cc + 7]));
        }
        tmem_st_wait();
      }
      fence_before_sync();
      __syncthreads();

      // Two passes over the segment: pass 0 rebuilds the chunk-start states
      // (saving each as an fp16 tile), pass 1 walks the chunks in reverse.
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
#pragma unroll 1
        for (int step = 0; step < c1 - c0; ++step) {
          const int c = pass == 0 ? c0 + step : c1 - 1 - step;
          const bool rev = pass == 1;
          uint4* slot = scratch + static_cast<size_t>(c - c0) * (32768 / 16);
          if (!rev) {
            for (int x = tid; x < 32768 / 16; x += kT) slot[x] = reinterpret_cast<const uint4*>(sm + OFF_A1)[x];
            if (c == c1 - 1) break;
          } else {
            for (int x = tid; x < 32768 / 16; x += kT) reinterpret_cast<uint4*>(sm + OFF_A1)[x] = slot[x];
          }
          const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
          const int rows = static_cast<int>(min(static_cast<int64_t>(kC), eos - t0));

          // ================= chunk prologue =================
          if (tid < kC) S[S_BETA + tid] = tid < rows ? sigm(bf(a.b + (t0 + tid) * a.H + h)) : 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = 8 * rh + j;
            const bool ok = r < rows;
            const int64_t off = ((t0 + r) * a.H + h) * kD + ci;
            QG[r * kLd + ci] = ok ? bf(a.q + off) : 0.f;
            KG[r * kLd + ci] = ok ? bf(a.k + off) : 0.f;
            VT[r * kLd + ci] = ok ? bf(a.v + off) : 0.f;
            GS[r * kLd + ci] = ok ? bf(a.g + off) : 0.f;
            if (rev) DOT[r * kLd + ci] = ok ? bf(a.dO + off) : 0.f;
          }
          __syncthreads();
          {  // row norms: warp w -> rows 2w, 2w+1
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int r = 2 * warp + rr;
              float sq = 0.f, sk = 0.f;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x = QG[r * kLd + lane + 32 * e], y = KG[r * kLd + lane + 32 * e];
                sq += x * x;
                sk += y * y;
              }
              sq = warp_sum(sq);
              sk = warp_sum(sk);
              if (lane == 0) {
                const float nq = sqrtf(sq + a.eps), nk = sqrtf(sk + a.eps);
                S[S_IQ0 + r] = nq > 0.f ? 1.f / nq : 0.f;
                S[S_IK0 + r] = nk > 0.f ? 1.f / nk : 0.f;
              }
            }
          }
          {  // gate, per-half cumulative log2 decay
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              const float d = r < rows ? Lg * sigm(expA * (GS[r * kLd + ci] + dtb)) : 0.f;
              acc += d;
              GS[r * kLd + ci] = acc;
            }
            S[S_TOT + rh * 128 + ci] = acc;
          }
          __syncthreads();
          {  // full cumsum, gated operands
            const float carry = rh ? S[S_TOT + ci] : 0.f;
            const float gend = S[S_TOT + ci] + S[S_TOT + 128 + ci];
            if (rh == 0) S[S_GEND + ci] = gend;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              const float G = GS[r * kLd + ci] + carry;
              GS[r * kLd + ci] = G;
              const float e = ex2(G), ei = ex2(-G);
              const float qh = QG[r * kLd + ci] * S[S_IQ0 + r] * a.scale;
              const float kh = KG[r * kLd + ci] * S[S_IK0 + r];
              const float kb = kh * ex2(gend - G);
              QG[r * kLd + ci] = qh * e;
              KG[r * kLd + ci] = kh * e;
              KI[r * kLd + ci] = kh * ei;
              KB[r * kLd + ci] = kb;
              st_h(sm + OFF_FKB, sw128_off(r, ci, 16), kb);
              if (rev) {
                st_h(sm + OFF_FQG, sw128_off(r, ci, 16), qh * e);
                st_h(sm + OFF_FDO, sw128_off(r, ci, 16), DOT[r * kLd + ci]);  // bf16 -> fp16 is exact
              }
            }
          }
          __syncthreads();
          // ================= intra-chunk matrices (fp32) =================
          {
            const int r = sr, s = ss;
            float aa = 0.f, am = 0.f;
            if (s <= r) {
#pragma unroll 8
              for (int i = 0; i < kD; ++i) {
                const float ki = KI[s * kLd + i];
                aa += KG[r * kLd + i] * ki;
                am += QG[r * kLd + i] * ki;
              }
            }
            S[S_AB + r * kSq + s] = s < r ? aa : 0.f;
            S[S_AQK + r * kSq + s] = s <= r ? am : 0.f;
            if (rev) {
              const float mv = s <= r ? am : 0.f;
              st_h(sm + OFF_FM, sw128_off(s, r, 16), mv);  // K-major B of dU~^T: row s, column r
              st_h(sm + OFF_FML, sw128_off(s, r, 16), lo_part(mv));
            }
          }
          __syncthreads();
          if (warp == 0) {  // T = (I + diag(beta) Abar)^-1, lane j: column j
            const int j = lane;
            float col[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
              float v = (r == j) ? 1.f : 0.f;
              if (r > j && j < 16) {
                const float br = S[S_BETA + r];
#pragma unroll
                for (int s = 0; s < r; ++s)
                  if (s >= j) v -= br * S[S_AB + r * kSq + s] * col[s];
              }
              col[r] = v;
              if (j < 16) {
                S[S_T + r * kSq + j] = v;
                S[S_TP + r * kSq + j] = v * S[S_BETA + j];
              }
            }
          }
          __syncthreads();
          {  // W = T' (Kh Gamma), U = T' V
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              float w = 0.f, u = 0.f;
#pragma unroll
              for (int s = 0; s < 16; ++s) {
                if (s <= r) {
                  const float t = S[S_TP + r * kSq + s];
                  w += t * KG[s * kLd + ci];
                  u += t * VT[s * kLd + ci];
                }
              }
              WT[r * kLd + ci] = w;
              UT[r * kLd + ci] = u;
              st_h(sm + OFF_FW, sw128_off(r, ci, 16), -w);
            }
          }
          fence_async_smem();
          fence_before_sync();
          KDA_SYNC_OR_BAIL();
          // ================= U~ = U - W H (tensor cores) =================
          if (tid == 0) {
            fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma(tmem + TM_D1, desc_kmajor(sb + OFF_A1, 128, 0, ks), desc_kmajor(sb + OFF_FW, 16, 0, ks),
                  idesc(128, 16), ks > 0);
            mma_commit(bar);
          }
          KDA_WAIT_MMA();
          fence_after_sync();
          {
            float x[8];
            tmem_ld8(tmem + tlane + TM_D1 + 8 * hh, x);  // lane = v, columns r
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * hh + j;
              const float u = UT[r * kLd + L] + x[j];
              UT[r * kLd + L] = u;
              st_h(sm + OFF_FU, sw128_off(r, L, 16), u);
            }
          }
          fence_async_smem();
          fence_before_sync();
          KDA_SYNC_OR_BAIL();

          if (!rev) {
            // ============ rebuild pass: H <- diag(gamma) H + Kbar^T U~ ============
            if (tid == 0) {
              fence_after_sync();
              mma(tmem + TM_D2, desc_mnmajor(sb + OFF_FU, 2048, 0), desc_mnmajor(sb + OFF_FKB, 2048, 0),
                  idesc(128, 128, true, true), 0);
              mma_commit(bar);
            }
            KDA_WAIT_MMA();
            fence_after_sync();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float hv[32], dv[32];
              tmem_ld32(tmem + tlane + TM_H + 64 * hh + 32 * half, hv);
              tmem_ld32(tmem + tlane + TM_D2 + 64 * hh + 32 * half, dv);
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int i = 64 * hh + 32 * half + j;
                hv[j] = ex2(S[S_GEND + i]) * hv[j] + dv[j];
              }
              tmem_st32(tmem + tlane + TM_H + 64 * hh + 32 * half, hv);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<uint4*>(sm + OFF_A1 + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)) =
                    make_uint4(pack_h2(hv[8 * cc], hv[8 * cc + 1]), pack_h2(hv[8 * cc + 2], hv[8 * cc + 3]),
                               pack_h2(hv[8 * cc + 4], hv[8 * cc + 5]), pack_h2(hv[8 * cc + 6], hv[8 * cc + 7]));
            }
            tmem_st_wait();
            fence_async_smem();
            fence_before_sync();
            KDA_SYNC_OR_BAIL();
            continue;
          }

          // ================= reverse pass: backward of chunk c =================
          // dU~^T = dO^T (Mhi + Mlo) + dH'^T Kbar^T
          if (tid == 0) {
            fence_after_sync();
            mma(tmem + TM_DU, desc_mnmajor(sb + OFF_FDO, 2048, 0), desc_kmajor(sb + OFF_FM, 16, 0, 0),
                idesc(128, 16, true, false), 0);
            mma(tmem + TM_DU, desc_mnmajor(sb + OFF_FDO, 2048, 0), desc_kmajor(sb + OFF_FML, 16, 0, 0),
                idesc(128, 16, true, false), 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma(tmem + TM_DU, desc_kmajor(sb + OFF_A1D, 128, 0, ks), desc_kmajor(sb + OFF_FKB, 16, 0, ks),
                  idesc(128, 16), 1);
            mma_commit(bar);
          }
          KDA_WAIT_MMA();
          fence_after_sync();
          {
            float x[8];
            tmem_ld8(tmem + tlane + TM_DU + 8 * hh, x);  // lane = v, columns r
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * hh + j;
              DUT[r * kLd + L] = x[j];
              st_h(sm + OFF_FDU, sw128_off(r, L, 16), x[j]);
            }
          }
          fence_async_smem();
          fence_before_sync();
          KDA_SYNC_OR_BAIL();
          if (tid == 0) {
            fence_after_sync();
            // state increment (Qh Gamma)^T dO - W^T dU~, transposed: dO^T QG + dU~^T (-W)
            mma(tmem + TM_D2, desc_mnmajor(sb + OFF_FDO, 2048, 0), desc_mnmajor(sb + OFF_FQG, 2048, 0),
                idesc(128, 128, true, true), 0);
            mma(tmem + TM_D2, desc_mnmajor(sb + OFF_FDU, 2048, 0), desc_mnmajor(sb + OFF_FW, 2048, 0),
                idesc(128, 128, true, true), 1);
            // (H dO^T), (H dU~^T), (dH' U~^T): lanes = key index i
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              mma(tmem + TM_DQ, desc_mnmajor(sb + OFF_A1, 16384, ks), desc_kmajor(sb + OFF_FDO, 16, 0, ks),
                  idesc(128, 16, true, false), ks > 0);
              mma(tmem + TM_DW, desc_mnmajor(sb + OFF_A1, 16384, ks), desc_kmajor(sb + OFF_FDU, 16, 0, ks),
                  idesc(128, 16, true, false), ks > 0);
              mma(tmem + TM_DK, desc_mnmajor(sb + OFF_A1D, 16384, ks), desc_kmajor(sb + OFF_FU, 16, 0, ks),
                  idesc(128, 16, true, false), ks > 0);
            }
            mma_commit(bar);
          }
          KDA_WAIT_MMA();
          fence_after_sync();
          // ---- dH update, dgamma (lane = v); dQG, dW, dKbar (lane = i) ----
          {
            float p[64];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float dh[32], inc[32];
              tmem_ld32(tmem + tlane + TM_DH + 64 * hh + 32 * half, dh);
              tmem_ld32(tmem + tlane + TM_D2 + 64 * hh + 32 * half, inc);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const uint4 hw = *reinterpret_cast<const uint4*>(sm + OFF_A1 + sw128_chunk(L, 8 * hh + 4 * half + cc, 128));
                const uint32_t hu[4] = {hw.x, hw.y, hw.z, hw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hu[e]));
                  p[32 * half + 8 * cc + 2 * e] = hf.x * dh[8 * cc + 2 * e];
                  p[32 * half + 8 * cc + 2 * e + 1] = hf.y * dh[8 * cc + 2 * e + 1];
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int i = 64 * hh + 32 * half + j;
                dh[j] = ex2(S[S_GEND + i]) * dh[j] + inc[j];
              }
              tmem_st32(tmem + tlane + TM_DH + 64 * hh + 32 * half, dh);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<uint4*>(sm + OFF_A1D + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)) =
                    make_uint4(pack_h2(dh[8 * cc], dh[8 * cc + 1]), pack_h2(dh[8 * cc + 2], dh[8 * cc + 3]),
                               pack_h2(dh[8 * cc + 4], dh[8 * cc + 5]), pack_h2(dh[8 * cc + 6], dh[8 * cc + 7]));
            }
            tmem_st_wait();
            // dgamma_i = sum_v H[i][v] dH'[i][v]: reduce the 64 products over the warp's lanes
            warp_reduce_scatter64(p, lane);
            {
              const int base = 32 * ((lane >> 4) & 1) + 16 * ((lane >> 3) & 1) + 8 * ((lane >> 2) & 1) +
                               4 * ((lane >> 1) & 1) + 2 * (lane & 1);
              S[S_RED + q4 * 128 + 64 * hh + base] = p[0];
              S[S_RED + q4 * 128 + 64 * hh + base + 1] = p[1];
            }
            float xq[8], xw[8], xk[8];
            tmem_ld8(tmem + tlane + TM_DQ + 8 * hh, xq);  // lane = i, columns r
            tmem_ld8(tmem + tlane + TM_DW + 8 * hh, xw);
            tmem_ld8(tmem + tlane + TM_DK + 8 * hh, xk);
            const int i = L;
            const float gend = S[S_GEND + i];
            float part = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * hh + j;
              const float G = GS[r * kLd + i];
              const float kbv = KB[r * kLd + i];
              AQ[r * kLd + i] = xq[j] * ex2(G);
              AG[r * kLd + i] = xq[j] * QG[r * kLd + i] - xk[j] * kbv;
              AK[r * kLd + i] = xk[j] * ex2(gend - G);
              WT[r * kLd + i] = -xw[j];  // dW (W itself is no longer needed)
              part += xk[j] * kbv;
            }
            S[S_PART + hh * 128 + i] = part;
          }
          __syncthreads();
          if (tid < kD) {  // d(chunk-end log decay) of channel tid
            const int i = tid;
            const float dgam = S[S_RED + i] + S[S_RED + 128 + i] + S[S_RED + 256 + i] + S[S_RED + 384 + i];
            S[S_DGE + i] = S[S_PART + i] + S[S_PART + 128 + i] + dgam * ex2(S[S_GEND + i]);
          }
          {  // dM = tril(dO U~^T), dT' = dW (Kh Gamma)^T + dU~ V^T
            const int r = sr, s = ss;
            float dm = 0.f, dt = 0.f;
#pragma unroll 8
            for (int i = 0; i < kD; ++i) {
              dm += DOT[r * kLd + i] * UT[s * kLd + i];
              dt += WT[r * kLd + i] * KG[s * kLd + i] + DUT[r * kLd + i] * VT[s * kLd + i];
            }
            S[S_DM + r * kSq + s] = s <= r ? dm : 0.f;
            S[S_DTP + r * kSq + s] = dt;
          }
          __syncthreads();
          {  // dV = T'^T dU~ (output), d(Kh Gamma) += T'^T dW
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              float dvv = 0.f, dkg = 0.f;
#pragma unroll
              for (int s = 0; s < 16; ++s) {
                if (s >= r) {
                  const float t = S[S_TP + s * kSq + r];
                  dvv += t * DUT[s * kLd + ci];
                  dkg += t * WT[s * kLd + ci];
                }
              }
              if (r < rows) a.dv[((t0 + r) * a.H + h) * kD + ci] = __float2bfloat16_rn(dvv);
              const float G = GS[r * kLd + ci];
              AK[r * kLd + ci] += dkg * ex2(G);
              AG[r * kLd + ci] += dkg * KG[r * kLd + ci];
            }
          }
          {  // dbeta from T' = T diag(beta); Y = (dT' diag(beta)) T^T
            const int r = sr, s = ss;
            if (tid < kC) {
              float db = 0.f;
#pragma unroll
              for (int r2 = 0; r2 < 16; ++r2) db += S[S_T + r2 * kSq + tid] * S[S_DTP + r2 * kSq + tid];
              S[S_DB + tid] = db;
            }
            float y = 0.f;
#pragma unroll
            for (int b2 = 0; b2 < 16; ++b2)
              if (b2 < r && b2 <= s) y += S[S_DTP + r * kSq + b2] * S[S_BETA + b2] * S[S_T + s * kSq + b2];
            S[S_Y + r * kSq + s] = y;
          }
          __syncthreads();
          {  // dA = -(T^T Y) strictly lower; dAbar = diag(beta) dA
            const int r = sr, s = ss;
            float da = 0.f;
            if (s < r) {
#pragma unroll
              for (int a2 = 0; a2 < 16; ++a2)
                if (a2 >= r) da -= S[S_T + a2 * kSq + r] * S[S_Y + a2 * kSq + s];
            }
            S[S_DA + r * kSq + s] = da;
          }
          __syncthreads();
          if (tid < kC) {  // dbeta of rows: A = diag(beta) Abar
            const int r = tid;
            float db = S[S_DB + r];
#pragma unroll
            for (int s = 0; s < 16; ++s)
              if (s < r) db += S[S_DA + r * kSq + s] * S[S_AB + r * kSq + s];
            S[S_DB + r] = db;
          }
          {  // Abar and M gradients back to kh, qh, G
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              const float br = S[S_BETA + r];
              float a1 = 0.f, a2 = 0.f, m1 = 0.f, m2 = 0.f;
#pragma unroll
              for (int s = 0; s < 16; ++s) {
                const float kis = KI[s * kLd + ci];
                if (s < r) a1 += S[S_DA + r * kSq + s] * kis;
                if (s > r) a2 += S[S_BETA + s] * S[S_DA + s * kSq + r] * KG[s * kLd + ci];
                if (s <= r) m1 += S[S_DM + r * kSq + s] * kis;
                if (s >= r) m2 += S[S_DM + s * kSq + r] * QG[s * kLd + ci];
              }
              a1 *= br;
              const float G = GS[r * kLd + ci], e = ex2(G), ei = ex2(-G);
              AQ[r * kLd + ci] += m1 * e;
              AK[r * kLd + ci] += a1 * e + (a2 + m2) * ei;
              AG[r * kLd + ci] += a1 * KG[r * kLd + ci] + m1 * QG[r * kLd + ci] - (a2 + m2) * KI[r * kLd + ci];
            }
          }
          __syncthreads();
          {  // dG of the chunk end, reverse cumulative sum (natural-log units)
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) sum += AG[(8 * rh + j) * kLd + ci];
            S[S_TOT + rh * 128 + ci] = sum;
          }
          __syncthreads();
          {
            float acc = S[S_DGE + ci] + (rh == 0 ? S[S_TOT + 128 + ci] : 0.f);
#pragma unroll
            for (int j = 7; j >= 0; --j) {
              const int r = 8 * rh + j;
              acc += AG[r * kLd + ci];
              AG[r * kLd + ci] = acc;
            }
          }
          {  // L2-norm chain rule row dots: warp w -> rows 2w, 2w+1
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int r = 2 * warp + rr;
              float sq = 0.f, sk = 0.f;
              if (r < rows) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int i = lane + 32 * e;
                  const int64_t off = ((t0 + r) * a.H + h) * kD + i;
                  sq += bf(a.q + off) * S[S_IQ0 + r] * AQ[r * kLd + i];
                  sk += bf(a.k + off) * S[S_IK0 + r] * AK[r * kLd + i];
                }
              }
              sq = warp_sum(sq);
              sk = warp_sum(sk);
              if (lane == 0) {
                S[S_RQ + r] = a.scale * sq;
                S[S_RK + r] = sk;
              }
            }
          }
          __syncthreads();
          {  // outputs dq, dk, dg (raw gate), parameter partials
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              if (r < rows) {
                const int64_t off = ((t0 + r) * a.H + h) * kD + ci;
                const float iq0 = S[S_IQ0 + r], ik0 = S[S_IK0 + r];
                const float xq = bf(a.q + off) * iq0, xk = bf(a.k + off) * ik0;
                a.dq[off] = __float2bfloat16_rn((a.scale * AQ[r * kLd + ci] - xq * S[S_RQ + r]) * iq0);
                a.dk[off] = __float2bfloat16_rn((AK[r * kLd + ci] - xk * S[S_RK + r]) * ik0);
                const float z = expA * (bf(a.g + off) + dtb);
                const float sg = sigm(z);
                const float dz = AG[r * kLd + ci] * a.lower * sg * (1.f - sg);
                a.dg[off] = __float2bfloat16_rn(expA * dz);
                acc_dtb += expA * dz;
                acc_alog += dz * z;
              }
            }
            if (tid < kC && tid < rows) {
              const float bt = S[S_BETA + tid];
              a.db[(t0 + tid) * a.H + h] = __float2bfloat16_rn(S[S_DB + tid] * bt * (1.f - bt));
            }
          }
          fence_async_smem();
          fence_before_sync();
          KDA_SYNC_OR_BAIL();
        }
        __syncthreads();
      }
    }
    // ---- per-(sequence, head) partial sums of the gate-parameter gradients ----
    S[S_RED + tid] = acc_dtb;
    __syncthreads();
    if (tid < kD) a.partial[static_cast<int64_t>(item) * (kD + 1) + tid] = S[S_RED + tid] + S[S_RED + 128 + tid];
    __syncthreads();
    S[S_RED + tid] = acc_alog;
    __syncthreads();
    for (int st = kT / 2; st > 0; st >>= 1) {
      if (tid < st) S[S_RED + tid] += S[S_RED + tid + st];
      __syncthreads();
    }
    if (tid == 0) a.partial[static_cast<int64_t>(item) * (kD + 1) + kD] = S[S_RED];
    __syncthreads();
  }
#undef KDA_WAIT_MMA
#undef KDA_SYNC_OR_BAIL
teardown:
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

__global__ void kda_param_reduce_tc_kernel(const float* partial, int N, int H, int D, float* dA_log, float* ddt_bias) {
  const int h = blockIdx.x;
  for (int i = threadIdx.x; i <= D; i += blockDim.x) {
    float s = 0.f;
    for (int n = 0; n < N; ++n) s += partial[(static_cast<int64_t>(n) * H + h) * (D + 1) + i];
    if (i < D)
      ddt_bias[h * D + i] = s;
    else
      dA_log[h] = s;
  }
}

}  // namespace

size_t bwd_scratch_bytes_per_cta_tc() { return static_cast<size_t>(kCPS) * 32768; }

kda_status launch_bwd_tc(const kda_problem* p, const BwdArgs& a, cudaStream_t s, int ctas) {
  if (p->head_dim != kD || p->dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;
  TcBwdArgs t;
  t.q = static_cast<const __nv_bfloat16*>(a.q);
  t.k = static_cast<const __nv_bfloat16*>(a.k);
  t.v = static_cast<const __nv_bfloat16*>(a.v);
  t.g = static_cast<const __nv_bfloat16*>(a.g);
  t.b = static_cast<const __nv_bfloat16*>(a.b);
  t.dO = static_cast<const __nv_bfloat16*>(a.dO);
  t.A_log = a.A_log;
  t.dt_bias = a.dt_bias;
  t.ckpt = a.ckpt;
  t.dq = static_cast<__nv_bfloat16*>(a.dq);
  t.dk = static_cast<__nv_bfloat16*>(a.dk);
  t.dv = static_cast<__nv_bfloat16*>(a.dv);
  t.dg = static_cast<__nv_bfloat16*>(a.dg);
  t.db = static_cast<__nv_bfloat16*>(a.db);
  t.partial = a.partial;
  t.scratch = reinterpret_cast<uint4*>(a.scratch);
  t.status = a.status;
  t.cu = a.cu;
  t.N = a.N;
  t.H = a.H;
  t.scale = a.scale;
  t.lower = a.lower;
  t.eps = a.eps;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  if (cudaFuncSetAttribute(kda_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (ctas > 0) kda_bwd_tc_kernel<<<ctas, kT, SMEM_BYTES, s>>>(t);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  kda_param_reduce_tc_kernel<<<p->num_heads, 128, 0, s>>>(a.partial, p->num_seqs, p->num_heads, kD, a.dA_log,
                                                          a.ddt_bias);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
