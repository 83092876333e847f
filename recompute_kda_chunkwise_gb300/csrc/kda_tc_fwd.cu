// kda_tc_fwd.cu -- tcgen05 tensor-core KDA forward (bf16 inputs, D = K = V = 128,
// chunk C = 64), one CTA of 256 threads per (sequence, head).
//
// Chunk math ("KDA at the production shape ...", section 2.1 op table; the
// state recurrence of section 1.1), with G the chunk-local inclusive
// cumulative log-decay, Gamma = exp(G), gamma = Gamma at the chunk end:
//   Abar[r,s] = sum_i kh_ri kh_si e^{G_ri - G_si} (s < r),  M[r,s] likewise with qh (s <= r)
//   T = (I + diag(beta) Abar)^-1,  T' = T diag(beta)
//   W = T' (Kh*Gamma),  U = T' V,  U~ = U - W H,  O = (Qh*Gamma) H + M U~
//   H' = diag(gamma) H + Kbar^T U~,   Kbar[s,i] = kh_si e^{G_{C-1,i} - G_si}
// The state is kept transposed, H^T (V x D), so every tensor-core product has
// M = 128 with the value index v (or the key index i) on the TMEM lanes; the
// fp32 master state lives in registers (thread (v, half) holds
// H^T[v][64*half .. 64*half+63]).
//
// Precision. Outputs must match an fp64 reference to 2e-2 of their RMS in the
// max norm; bf16 operands (8-bit significands) miss that by 3-5x on these
// heavy-tailed outputs, fp16 operands (11-bit) meet it. Every tensor-core
// operand is therefore fp16 (bounded quantities: states, W, U~, T', M, gated
// q/k, Kbar, and V converted from bf16), except the factors of Abar and M:
// exp(G_r - G_s) spans e^{320} over 64 tokens at the -5 gate floor (section
// 3(a) of the same page: the inverse-decay factor of k leaves fp32 range once
// the cumulative log-decay passes -88, i.e. beyond 17 tokens at that floor), so
// Abar and M are built from four 16-token column blocks J, each referenced
// at the end of block J: the row operand kh_r e^{G_r - B_{J+1}} (rows
// r >= 16J, up to e^{80}) times the column operand kh_s e^{B_{J+1} - G_s}
// (s in block J, down to e^{-80}). Those factors need fp32 range, so the four
// 128 x 16 x 128 products run as kind::tf32 with the row operand written to
// TMEM (k rows on lanes 0-63, q rows on lanes 64-127).
//
// The O = M U~ term dominates the remaining error (the largest outputs are
// mostly intra-chunk), so M, U~ (in that product) and T' are carried as fp16
// hi + lo pairs and their products take three (M U~) or two (T' products)
// MMAs.
//
// Stages per chunk (sequential; every tcgen05 completion and TMA arrival is
// awaited on an mbarrier with a bounded wait): TMA of q, k, raw gate -> row
// norms -> gate and cumulative decay (channel-major) -> operand tiles
// (row-major) -> four tf32 rounds for Abar | M -> T by blocked forward
// substitution -> TMA'd V converted to fp16 -> W, U products -> -W tile ->
// H^T products -> U~^T tile -> Kbar, M products -> state update and output.
#include "kda_tc_common.cuh"

#ifdef KDA_STAGE_TIMERS
// per-CTA stage counters of the tensor-core forward (tracing build)
__device__ unsigned long long g_fwd_stage[kStageCtas * 32];
extern "C" int kda_fwd_stage_timers(unsigned long long* host, int clear) {
  static unsigned long long zero[kStageCtas * 32];
  if (host != nullptr && cudaMemcpyFromSymbol(host, g_fwd_stage, sizeof(g_fwd_stage)) != cudaSuccess) return 1;
  if (clear && cudaMemcpyToSymbol(g_fwd_stage, zero, sizeof(zero)) != cudaSuccess) return 1;
  return 0;
}
#endif

namespace kda {
namespace {
using namespace tc;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Stages of a chunk step, as the stage timers of a tracing build count them
// (each mark closes the stage named by it; FS_UPDATE, at the loop top, closes
// the previous chunk's state update and output).
enum FwdStage {
  FS_UPDATE,        // state update (fp32 registers), next H^T operand, output
  FS_TOP,           // loop top: next helper job / checkpoint store
  FS_QKG_WAIT,      // q / k / raw gate tiles landed (TMA)
  FS_NORMS,         // row norms (and a helper's wait for its previous stores)
  FS_GATE,          // gate, cumulative log2-decay
  FS_REFS,          // per-channel block references
  FS_OPERANDS,      // operand tiles
  FS_ROUNDS,        // Abar | M tf32 rounds (row operands to TMEM, four MMA rounds)
  FS_ROUND_READOUT, // Abar and M out of TMEM
  FS_INVERSE,       // T by blocked forward substitution
  FS_WU,            // v -> fp16, W / U products
  FS_NEG_W,         // -W tile
  FS_HANDOFF,       // helper: the prepared chunk's bulk stores issued
  FS_SLOT_WAIT,     // main CTA: a handed chunk's operands landed
  FS_UT_O,          // U~ and the H^T part of O (tcgen05)
  FS_KBAR_M,        // U~ tile, Kbar^T U~ and M U~ (tcgen05)
  FS_NEXT_SLOT,     // split mode: wait for, and fetch, the next handed chunk
  FS_COUNT
};
static_assert(FS_COUNT <= 31, "stage slots");

// Shared-memory map (bytes from a 1024-byte aligned base).
constexpr int OFF_STG_Q = 0;           // staged q        [64 r][128 c] bf16 SW128 (TMA)
constexpr int OFF_STG_K = 16384;       // staged k
constexpr int OFF_STG_G = 32768;       // staged raw gate
constexpr int OFF_A1 = 49152;          // H^T fp16 [128 v][128 i]
constexpr int OFF_B1 = 81920;          // [-W (64 r) ; Qh*Gamma (64 r)] x [128 i] fp16
constexpr int OFF_B2A = 114688;        // Kbar [64 r][128 i] fp16 (read MN-major)
constexpr int OFF_B2B = 131072;        // M [64 r][64 s] fp16
constexpr int OFF_XW = 139264;         // Kh*Gamma [64 s][128 i] fp16 (read MN-major); later U~^T [128 v][64 r]
constexpr int OFF_R = 155648;          // 64 KB, reused within a chunk:
constexpr int OFF_XS = OFF_R;          //   log2 offsets G_r - B_{I+1}, fp32 [64][128] (swizzled rows)
constexpr int OFF_BK = OFF_R + 32768;  //   column operands kh_s e^{B-G_s}, tf32 [64 s][128 i]
constexpr int OFF_TOT = OFF_R + 61440; //   block totals [4][128] fp32 (dead before BK is written)
constexpr int OFF_V = OFF_R;           //   then staged v (bf16 -> fp16 in place) [64 s][128 v]
constexpr int OFF_ABAR = OFF_R + 16384;//   then Abar fp32 [64][65]
constexpr int OFF_TF = OFF_R + 33024;  //        T fp32 [64][65]
constexpr int OFF_TP = OFF_R + 50176;  //        T' fp16 [64 r][64 s]
constexpr int OFF_X = OFF_R + 58368;   //        fp32 scratch [8][16][9]
constexpr int OFF_TPL = OFF_R + 16384; //   after the inverse (Abar dead): T' low part fp16 [64 r][64 s]
constexpr int OFF_ML = OFF_R + 24576;  //                                  M low part fp16 [64 r][64 s]
constexpr int OFF_UL = OFF_R;          //   after the U product (v dead): U~^T low part fp16 [128 v][64 r]
constexpr int OFF_WG = OFF_R + 33792;  //   GDN-2: after the inverse (T dead), the raw write gate bf16 SW128 [64 s][128 v]
constexpr int OFF_SMALL = OFF_R + 65536;
// small fp32 arrays
constexpr int SM_BETA = 0, SM_IQ = 64, SM_IK = 128, SM_GAM = 192, SM_EB = 320, SM_EK = 832, SM_U = 1344;
constexpr int SM_GAM2 = 1344 + 6 * 128;  // gamma of a handed-over chunk (split mode)
constexpr int SMALL_FLOATS = SM_GAM2 + 128;
constexpr int OFF_BAR = OFF_SMALL + SMALL_FLOATS * 4;
constexpr int SMEM_USED = OFF_BAR + 80;  // 10 mbarrier / flag words
constexpr int OFF_STAGE = SMEM_USED;  // stage counters (tracing build only)
constexpr int SMEM_BYTES = SMEM_USED + KDA_STAGE_BYTES + 1024;  // alignment slack

// Split-mode hand-off slot (bytes, all 16-byte multiples): the prepared
// operands of one odd chunk as the main CTA's shared memory holds them, in
// two contiguous runs of that memory plus T' hi and gamma. The main CTA forms
// U^T = V^T T'^T itself, in the product that also accumulates H^T (-W)^T.
constexpr uint32_t kXB = 0;                       // OFF_B1..OFF_XW: [-W ; Qh*Gamma] | Kbar | M hi, 56 KB
constexpr uint32_t kXBBytes = OFF_XW - OFF_B1;
constexpr uint32_t kXR = kXB + kXBBytes;          // OFF_V..: v fp16 | T' lo | M lo, 32 KB
constexpr uint32_t kXRBytes = OFF_ML + 8192 - OFF_V;
constexpr uint32_t kXTP = kXR + kXRBytes;         // T' hi fp16, 8 KB (OFF_TP)
constexpr uint32_t kXGAM = kXTP + 8192;           // gamma [128] fp32
constexpr uint32_t kXSlotBytes = kXGAM + 512;
static_assert(OFF_B2A == OFF_B1 + 32768 && OFF_B2B == OFF_B2A + 16384 && OFF_XW == OFF_B2B + 8192, "slot run B");
static_assert(OFF_TPL == OFF_V + 16384 && OFF_ML == OFF_TPL + 8192, "slot run R");
constexpr int kXSlots = 4;                        // ring depth per item

// TMEM columns
constexpr uint32_t TM_DA = 0;    // Abar (lanes 0-63) | M (lanes 64-127), 64 columns
constexpr uint32_t TM_DW = 64;   // W^T (lanes = i), 64 columns
constexpr uint32_t TM_DU = 128;  // U~^T, 64 columns
constexpr uint32_t TM_DO = 192;  // O^T, 64 columns
constexpr uint32_t TM_DH = 256;  // (Kbar^T U~)^T, 128 columns
constexpr uint32_t TM_AJ = 64;   // tf32 row operands of the Abar | M rounds: rounds 0..2 at
                                 // 64 + 128 J (columns free until the W/U products), round 3
                                 // reuses round 0's columns
constexpr uint32_t TM_COLS = 512;

struct TcFwdArgs {
  const __nv_bfloat16* b;
  const float* A_log;
  const float* dt_bias;
  __nv_bfloat16* o;
  const float* h0;  // initial states [N][H][D][D] (NULL: zero)
  float* hT;        // final states (NULL: not written)
  float* ckpt;
  int* status;
  const int32_t* cu;
  int64_t S;  // total tokens (cu[N])
  int N, H;
  float scale, lower, eps;
  int test_timeout;
  // split mode (helpers > 0): CTAs N*H .. N*H+helpers-1 prepare the odd
  // chunks of every item and hand them over through xbuf / xflags
  int helpers;
  uint32_t* xflags;  // per item: [4] last odd-chunk index + 1 written into slot q, [4] consumed count
  uint8_t* xbuf;     // per item: kXSlots slots of kXSlotBytes
};

__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + ex2(-x * kLog2e)); }

// fp32 [64][128] tile with 16-byte chunks XOR-swizzled by row (conflict-free
// row and column walks).
__device__ __forceinline__ uint32_t xs_off(int r, int c) {
  return static_cast<uint32_t>(r * 512 + (c >> 5) * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + ((c & 3) << 2));
}

// T = (I + N)^-1, N = diag(beta) Abar strictly lower (fp32; the Abar tile
// already holds N, rows scaled when it is written), in 16 x 16 blocks:
//  * each diagonal block by one warp, itself in 8 x 8 halves: lane j < 16
//    solves column j of its half by right-looking forward substitution, then
//    lanes 0-7 form the lower-left 8 x 8 part as -T22 N21 T11;
//  * T_10 and T_32 = -T_II N_IJ T_JJ (level A), then the lower-left 32 x 32
//    part as -T_hi (N_21 T_lo) in two product phases on all eight warps;
// products on warp-level tf32 tiles split into hi + lo parts (about fp32
// accuracy); finally T' = T diag(beta) as fp16 hi + lo parts.
__device__ __forceinline__ void tri_inverse(uint8_t* sm, const float* s_beta, int tid) {
  float* Ab = reinterpret_cast<float*>(sm + OFF_ABAR);
  float* Tf = reinterpret_cast<float*>(sm + OFF_TF);
  float* X = reinterpret_cast<float*>(sm + OFF_X);
  const int warp = tid >> 5, lane = tid & 31, fg = lane >> 2, ft = lane & 3;
  if (warp < 4) {
    const int base = 16 * warp, j = lane & 15, b8 = 8 * (j >> 3);
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (b8 + k == j) ? 1.f : 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 7; ++s2) {
#pragma unroll
      for (int k = s2 + 1; k < 8; ++k) x[k] -= Ab[(base + b8 + k) * 65 + base + b8 + s2] * x[s2];
    }
    if (lane < 16) {
#pragma unroll
      for (int k = 0; k < 8; ++k) Tf[(base + b8 + k) * 65 + base + j] = x[k];
    }
    __syncwarp();
    float z[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) z[k] = 0.f;
    if (lane < 8) {
      float y[8];  // (N21 T11)[., j] within the block
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float acc = 0.f;
#pragma unroll
        for (int s3 = 0; s3 < 8; ++s3) acc += Ab[(base + 8 + k) * 65 + base + s3] * x[s3];
        y[k] = acc;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m <= k; ++m) acc += Tf[(base + 8 + k) * 65 + base + 8 + m] * y[m];
        z[k] = -acc;
      }
    }
    if (lane < 16) {
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const float t = ((r >> 3) == (j >> 3)) ? x[r & 7] : ((r >= 8) ? z[r - 8] : 0.f);
        Tf[(base + r) * 65 + base + j] = t;
      }
    }
  } else {  // the six blocks above the diagonal are zero
    for (int x = tid - 128; x < 6 * 256; x += 128) {
      const int b = x >> 8, e = x & 255;
      const int I = b < 3 ? 0 : (b < 5 ? 1 : 2), J = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
      Tf[(16 * I + (e >> 4)) * 65 + 16 * J + (e & 15)] = 0.f;
    }
  }
  __syncthreads();
  // product of a 16-row block tile (A: 16 x 16 at A0, stride lda) with this
  // warp's 8 columns of B (16 x 8 at B0, stride ldb), accumulated into acc
  auto mma_block = [&](float (&acc)[4], const float* A0, int lda, const float* B0, int ldb) {
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
      float fa[4], fb[2];
      ldA(fa, A0, lda, k0, fg, ft);
      ldBr(fb, B0, ldb, 0, k0, fg, ft);
      mma3(acc, fa, fb);
    }
  };
  auto store_tile = [&](float* dst, int ld, const float (&v)[4], float sgn) {
    dst[fg * ld + 2 * ft] = sgn * v[0];
    dst[fg * ld + 2 * ft + 1] = sgn * v[1];
    dst[(fg + 8) * ld + 2 * ft] = sgn * v[2];
    dst[(fg + 8) * ld + 2 * ft + 1] = sgn * v[3];
  };
  // level A: T_10 and T_32 (warps 0-3: block J = 2 (w >> 1), 8-column half nt)
  if (warp < 4) {
    const int J = 2 * (warp >> 1), I = J + 1, nt = warp & 1;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    mma_block(acc, Ab + (16 * I) * 65 + 16 * J, 65, Tf + (16 * J) * 65 + 16 * J + 8 * nt, 65);
    float* Xw = X + warp * (16 * 9);  // N_IJ T_JJ, this warp's 8 columns
    store_tile(Xw, 9, acc, 1.f);
    __syncwarp();
    float t2[4] = {0.f, 0.f, 0.f, 0.f};
    mma_block(t2, Tf + (16 * I) * 65 + 16 * I, 65, Xw, 9);
    store_tile(Tf + (16 * I) * 65 + 16 * J + 8 * nt, 65, t2, -1.f);
  }
  __syncthreads();
  // level B: Y_IJ = sum_{K=J..1} N_IK T_KJ for I in {2, 3}, J in {0, 1}
  // (warp w: I = 2 + (w >> 2), J = (w >> 1) & 1, half nt = w & 1)
  const int I = 2 + (warp >> 2), J = (warp >> 1) & 1, nt = warp & 1;
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int K = J; K < 2; ++K)
      mma_block(acc, Ab + (16 * I) * 65 + 16 * K, 65, Tf + (16 * K) * 65 + 16 * J + 8 * nt, 65);
    store_tile(X + warp * (16 * 9), 9, acc, 1.f);
  }
  __syncthreads();
  // T_IJ = -sum_{K=2..I} T_IK Y_KJ (Y_KJ: warp (K - 2) * 4 + J * 2 + nt's tile)
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int K = 2; K <= I; ++K)
      mma_block(acc, Tf + (16 * I) * 65 + 16 * K, 65, X + ((K - 2) * 4 + J * 2 + nt) * (16 * 9), 9);
    store_tile(Tf + (16 * I) * 65 + 16 * J + 8 * nt, 65, acc, -1.f);
  }
  __syncthreads();
  for (int x = tid; x < 64 * 32; x += kThreads) {
    const int r = x >> 5, s = 2 * (x & 31);
    const float t0 = Tf[r * 65 + s] * s_beta[s], t1 = Tf[r * 65 + s + 1] * s_beta[s + 1];
    const uint32_t hi = pack_h2(t0, t1);
    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    *reinterpret_cast<uint32_t*>(sm + OFF_TP + sw128_off(r, s, 64)) = hi;
    *reinterpret_cast<uint32_t*>(sm + OFF_TPL + sw128_off(r, s, 64)) = pack_h2(t0 - hf.x, t1 - hf.y);
  }
}

// CG: the GDN-2 operator (channel-wise erase gate on the key channels, write
// gate on the value channels, in place of beta): the erase gate scales the
// k rows of the Abar row operand and the Kh*Gamma operand of W, the write
// gate scales V before U = T (w * V), and T' = T. tme / tmw map the raw erase
// and write gates [S,H,D] (unused for KDA).
template <bool CG>
__global__ void __launch_bounds__(kThreads, 1)
    kda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmg,
                      const __grid_constant__ CUtensorMap tme, const __grid_constant__ CUtensorMap tmw,
                      const TcFwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(sm);
  const uint64_t D0 = sdesc(sb, 0);  // base of every tcgen05 shared-memory descriptor
  float* smf = reinterpret_cast<float*>(sm + OFF_SMALL);
  float* s_beta = smf + SM_BETA;
  float* s_iq = smf + SM_IQ;
  float* s_ik = smf + SM_IK;
  float* s_gam = smf + SM_GAM;
  float* s_eB = smf + SM_EB;  // [4][128]  2^{B_{I+1}}
  float* s_eK = smf + SM_EK;  // [4][128]  2^{G_end - B_{I+1}}
  float* s_u = smf + SM_U;    // [6][128]  2^{B_{I+1} - B_{J+1}}, pair I(I-1)/2 + J
  float* s_tot = reinterpret_cast<float*>(sm + OFF_TOT);
  uint64_t* bar_qkg = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_v = bar_qkg + 1;
  uint64_t* bar_mma = bar_qkg + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_qkg + 3);
  int* s_fail = reinterpret_cast<int*>(bar_qkg + 4);
  uint64_t* bar_odd = bar_qkg + 5;  // completion of Abar | M round 1
  uint64_t* bar_r2 = bar_qkg + 6;   // completion of Abar | M round 2
  uint64_t* bar_x = bar_qkg + 7;    // split mode: a handed-over odd chunk has landed
  uint64_t* bar_e = bar_qkg + 8;    // GDN-2: the erase-gate tile has landed
  uint64_t* bar_w = bar_qkg + 9;    // GDN-2: the write-gate tile has landed
  float* s_gam2 = smf + SM_GAM2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Roles. Without helpers, CTA b walks every chunk of item b. In split mode
  // the main CTA b < items prepares its even chunks itself and takes the odd
  // ones prepared by the helper CTAs, which walk jobs t * items + item (odd
  // chunk 2t + 1 of item) in order, helper j taking jobs j, j + helpers, ...
  const int items = a.N * a.H;
  const bool split = a.helpers > 0;
  const bool helper = split && static_cast<int>(blockIdx.x) >= items;
  int item = helper ? 0 : static_cast<int>(blockIdx.x);
  int n = item / a.H, h = item % a.H;
  int64_t bos = a.cu[n], eos = a.cu[n + 1];
  int nchunks = helper ? 0 : static_cast<int>((eos - bos + kC - 1) / kC);
  int job = static_cast<int>(blockIdx.x) - items, max_jobs = 0;
  if (helper) {
    int max_odd = 0;
    for (int s2 = 0; s2 < a.N; ++s2)
      max_odd = max(max_odd, static_cast<int>((a.cu[s2 + 1] - a.cu[s2] + kC - 1) / kC) / 2);
    max_jobs = max_odd * items;
  }

  if (tid == 0) {
    mbar_init(bar_qkg, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_odd, 1);
    mbar_init(bar_r2, 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_e, 1);
    mbar_init(bar_w, 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(s_tmem, TM_COLS);
  for (int x = tid; x < 32768 / 16; x += kThreads) reinterpret_cast<uint4*>(sm + OFF_A1)[x] = make_uint4(0, 0, 0, 0);
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *s_tmem;
  KDA_STAGE_INIT(sm + OFF_STAGE);

  // channel-major role: channel pair (c0, c0+1), rows 16*Ib .. 16*Ib+15 (sub-block Ib)
  const int pp = tid & 63, Ib = tid >> 6, c0 = 2 * pp;
  float expA = expf(a.A_log[h]);
  float dtb0 = a.dt_bias[h * kD + c0], dtb1 = a.dt_bias[h * kD + c0 + 1];
  const float Lg = a.lower * kLog2e;
  // lane roles: TMEM lane quarter q4, column half hh
  const int q4 = warp & 3, hh = warp >> 2, lrow = 32 * q4 + lane;
  const uint32_t tlane = static_cast<uint32_t>(32 * q4) << 16;
  // row-major role (operand tiles): k rows (q4 < 2) or q rows (q4 >= 2)
  const bool krole = q4 < 2;
  const int prow = 32 * (q4 & 1) + lane, pI = prow >> 4;
  float Hst[64];  // H[64 hh + j][lrow]
#pragma unroll
  for (int j = 0; j < 64; ++j) Hst[j] = 0.f;
  if (!helper && a.h0 != nullptr) {  // initial state: registers and its fp16 operand tile
    const float* src = a.h0 + static_cast<int64_t>(item) * (kD * kD);
#pragma unroll
    for (int j = 0; j < 64; ++j) Hst[j] = src[(64 * hh + j) * kD + lrow];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      *reinterpret_cast<uint4*>(sm + OFF_A1 + sw128_chunk(lrow, 8 * hh + cc, 128)) =
          make_uint4(pack_h2(Hst[8 * cc], Hst[8 * cc + 1]), pack_h2(Hst[8 * cc + 2], Hst[8 * cc + 3]),
                     pack_h2(Hst[8 * cc + 4], Hst[8 * cc + 5]), pack_h2(Hst[8 * cc + 6], Hst[8 * cc + 7]));
  }
  uint32_t ph_qkg = 0, ph_v = 0, ph_mma = 0, ph_odd = 0, ph_r2 = 0, ph_x = 0, ph_e = 0, ph_w = 0;
  bool x_pending = false;  // a hand-over load into shared memory is in flight

  auto issue_qkg = [&](int hd, int t) {
    mbar_expect_tx(bar_qkg, 6 * 8192);
    tma_load_3d(sm + OFF_STG_Q, &tmq, 0, hd, t, bar_qkg);
    tma_load_3d(sm + OFF_STG_Q + 8192, &tmq, 64, hd, t, bar_qkg);
    tma_load_3d(sm + OFF_STG_K, &tmk, 0, hd, t, bar_qkg);
    tma_load_3d(sm + OFF_STG_K + 8192, &tmk, 64, hd, t, bar_qkg);
    tma_load_3d(sm + OFF_STG_G, &tmg, 0, hd, t, bar_qkg);
    tma_load_3d(sm + OFF_STG_G + 8192, &tmg, 64, hd, t, bar_qkg);
  };
  auto issue_v = [&](int t) {
    mbar_expect_tx(bar_v, 2 * 8192);
    tma_load_3d(sm + OFF_V, &tmv, 0, h, t, bar_v);
    tma_load_3d(sm + OFF_V + 8192, &tmv, 64, h, t, bar_v);
  };
  auto issue_u = [&]() {  // U^T = V^T (T'hi + T'lo)^T
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma(tmem + TM_DU, desc_mn(D0, OFF_V, 8192, ks & 3), desc_k(D0, (ks < 4 ? OFF_TP : OFF_TPL), 64, 0, ks & 3),
          idesc(128, 64, true, false), ks > 0);
  };
#define KDA_WAIT(bar, ph)                                         \
  do {                                                            \
    if (!mbar_wait(bar, ph, a.status, wait_limit)) *s_fail = 1;   \
    ph ^= 1u;                                                     \
  } while (0)
#define KDA_SYNC_OR_BAIL()      \
  do {                          \
    __syncthreads();            \
    if (*s_fail) goto teardown; \
  } while (0)

  // (KDA_FLAG_TEST_TIMEOUT: the first load is skipped, so its short wait runs out)
  const int wait_limit = a.test_timeout ? (1 << 12) : (1 << 24);
  // a helper looks one job ahead, so that the next job's loads overlap this one
  int nx_item = 0, nx_c = -1;
  auto find_job = [&]() {
    nx_c = -1;
    while (job < max_jobs) {
      const int tt = job / items, it = job % items, s2 = it / a.H;
      job += a.helpers;
      if (2 * tt + 1 < static_cast<int>((a.cu[s2 + 1] - a.cu[s2] + kC - 1) / kC)) {
        nx_item = it;
        nx_c = 2 * tt + 1;
        return;
      }
    }
  };
  auto issue_next_job = [&]() {
    issue_qkg(nx_item % a.H, static_cast<int>(a.cu[nx_item / a.H] + static_cast<int64_t>(nx_c) * kC));
  };
  bool pub_pending = false;  // helper: a hand-off whose stores are in flight, not yet published
  int pub_item = 0, pub_tt = 0;
  auto publish = [&]() {  // thread 0 of a helper
    bulk_wait_all();
    fence_proxy_global();
    st_release(a.xflags + 5 * pub_item + pub_tt % kXSlots, static_cast<uint32_t>(pub_tt + 1));
  };
  if (helper) {
    find_job();
    if (tid == 0 && nx_c >= 0) issue_next_job();
  } else if (tid == 0 && nchunks > 0 && !a.test_timeout) {
    issue_qkg(h, static_cast<int>(bos));
  }

  int c = -1;
  while (true) {
    KDA_STAGE(FS_UPDATE);
    if (!helper) {
      if (++c >= nchunks) break;
    } else {  // the job found ahead, whose q, k, g are in flight
      if (nx_c < 0) break;
      item = nx_item;
      c = nx_c;
      n = item / a.H;
      h = item % a.H;
      bos = a.cu[n];
      eos = a.cu[n + 1];
      nchunks = static_cast<int>((eos - bos + kC - 1) / kC);
      expA = expf(a.A_log[h]);
      dtb0 = a.dt_bias[h * kD + c0];
      dtb1 = a.dt_bias[h * kD + c0 + 1];
      find_job();
    }
    KDA_STAGE(FS_TOP);
    KDA_STAGE_STEP();
    const bool handed = split && !helper && (c & 1);  // prepared by a helper
    const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kC), eos - t0));

    if (!helper && a.ckpt != nullptr && (c % (kCkptTokens / kC)) == 0) {
      float* dst = a.ckpt + (ckpt_slot(bos, n, c / (kCkptTokens / kC)) * a.H + h) * static_cast<int64_t>(kD * kD);
#pragma unroll
      for (int j = 0; j < 64; ++j) dst[(64 * hh + j) * kD + lrow] = Hst[j];
    }

    if (!handed) {
    // raw beta: loaded now, stored once the norms are done (its latency hidden)
    const unsigned short braw = (!CG && tid < rows) ? beta_bits(a.b, (t0 + tid) * a.H + h) : 0;
    KDA_WAIT(bar_qkg, ph_qkg);
    KDA_STAGE(FS_QKG_WAIT);
    // ---- row norms: warp w handles rows 8w .. 8w+7, four at a time (sums
    // interleaved; lanes 0-3 finish the q rows, lanes 8-11 the k rows) ----
#pragma unroll
    for (int b4 = 0; b4 < 2; ++b4) {
      float sq[4], sk[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int r = warp * 8 + 4 * b4 + rr;
        const uint2 qv = *reinterpret_cast<const uint2*>(sm + OFF_STG_Q + sw128_off(r, 4 * lane, 64));
        const uint2 kv = *reinterpret_cast<const uint2*>(sm + OFF_STG_K + sw128_off(r, 4 * lane, 64));
        const float2 q01 = unpack_bf16(qv.x), q23 = unpack_bf16(qv.y);
        const float2 k01 = unpack_bf16(kv.x), k23 = unpack_bf16(kv.y);
        sq[rr] = q01.x * q01.x + q01.y * q01.y + q23.x * q23.x + q23.y * q23.y;
        sk[rr] = k01.x * k01.x + k01.y * k01.y + k23.x * k23.x + k23.y * k23.y;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          sq[rr] += __shfl_xor_sync(0xffffffffu, sq[rr], o);
          sk[rr] += __shfl_xor_sync(0xffffffffu, sk[rr], o);
        }
      }
      float mine = sq[0];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        if ((lane & 3) == rr) mine = (lane & 8) ? sk[rr] : sq[rr];
      }
      if ((lane & 4) == 0 && lane < 16) {
        const int r = warp * 8 + 4 * b4 + (lane & 3);
        const bool ok = r < rows;
        const float nrm = sqrtf(mine + a.eps);
        if (lane & 8)
          s_ik[r] = (ok && nrm > 0.f) ? 1.f / nrm : 0.f;
        else
          s_iq[r] = (ok && nrm > 0.f) ? a.scale / nrm : 0.f;
      }
    }
    if (tid < kC)  // GDN-2: beta = 1 on every valid row (the gates act per channel)
      s_beta[tid] = tid < rows ? (CG ? 1.f : sigmoidf_(__bfloat162float(__ushort_as_bfloat16(braw)))) : 0.f;
    if (pub_pending) {  // the previous job's stores still read the region the offsets go to
      if (tid == 0) bulk_wait_read();
      __syncthreads();
    }
    KDA_STAGE(FS_NORMS);
    // ---- gate and cumulative log2-decay of the thread's 16-row block ----
    {
      float gl0[16], gl1[16], acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int r = 16 * Ib + j;
        const float2 g2 = unpack_bf16(*reinterpret_cast<const uint32_t*>(sm + OFF_STG_G + sw128_off(r, c0, 64)));
        const float d0 = r < rows ? Lg * sigmoid_fast(expA * (g2.x + dtb0)) : 0.f;
        const float d1 = r < rows ? Lg * sigmoid_fast(expA * (g2.y + dtb1)) : 0.f;
        acc0 += d0;
        acc1 += d1;
        gl0[j] = acc0;
        gl1[j] = acc1;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)  // G_r - B_{I+1} >= 0
        *reinterpret_cast<float2*>(sm + OFF_XS + xs_off(16 * Ib + j, c0)) = make_float2(gl0[j] - acc0, gl1[j] - acc1);
      s_tot[Ib * 128 + c0] = acc0;
      s_tot[Ib * 128 + c0 + 1] = acc1;
    }
    __syncthreads();
    if (CG && tid == 0) {  // the raw gate is consumed: the erase gate takes its tile
      mbar_expect_tx(bar_e, 2 * 8192);
      tma_load_3d(sm + OFF_STG_G, &tme, 0, h, static_cast<int>(t0), bar_e);
      tma_load_3d(sm + OFF_STG_G + 8192, &tme, 64, h, static_cast<int>(t0), bar_e);
    }
    KDA_STAGE(FS_GATE);
    // ---- per-channel block references ----
    if (tid < kD) {
      const int ch = tid;
      float B[5];
      B[0] = 0.f;
#pragma unroll
      for (int I = 0; I < 4; ++I) B[I + 1] = B[I] + s_tot[I * 128 + ch];
      s_gam[ch] = ex2(B[4]);
#pragma unroll
      for (int I = 0; I < 4; ++I) {
        s_eB[I * 128 + ch] = ex2(B[I + 1]);
        s_eK[I * 128 + ch] = ex2(B[4] - B[I + 1]);
#pragma unroll
        for (int J = 0; J < I; ++J) s_u[(I * (I - 1) / 2 + J) * 128 + ch] = ex2(B[I + 1] - B[J + 1]);
      }
    }
    __syncthreads();

    KDA_STAGE(FS_REFS);
    // ---- operand tiles, row-major: thread = one row (k or q) x 64 channels ----
    if (CG) KDA_WAIT(bar_e, ph_e);  // GDN-2: the erase gate (in the raw gate's tile)
    float rowf[64];  // kh e^{G_r - B_{I+1}} (k rows) or qh e^{G_r - B_{I+1}} (q rows)
    {
      // k rows build Kh*Gamma and Kbar, q rows build Qh*Gamma and the tf32 column
      // operand of the same token's k row (two exponentials each, balanced)
      const int r = prow;
      const float nrm = krole ? s_ik[r] : s_iq[r];
      const float nrmk = s_ik[r];
      const uint32_t src = krole ? OFF_STG_K : OFF_STG_Q;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int ch0 = 64 * hh + 8 * cc;
        const uint4 raw = *reinterpret_cast<const uint4*>(sm + src + sw128_chunk(r, 8 * hh + cc, 64));
        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
        uint4 rawk = raw;
        if (!krole) rawk = *reinterpret_cast<const uint4*>(sm + OFF_STG_K + sw128_chunk(r, 8 * hh + cc, 64));
        const uint32_t rk[4] = {rawk.x, rawk.y, rawk.z, rawk.w};
        uint32_t re[4] = {0u, 0u, 0u, 0u};  // GDN-2, k rows: the raw erase gate of these channels
        if (CG && krole) {
          const uint4 rawe = *reinterpret_cast<const uint4*>(sm + OFF_STG_G + sw128_chunk(r, 8 * hh + cc, 64));
          re[0] = rawe.x; re[1] = rawe.y; re[2] = rawe.z; re[3] = rawe.w;
        }
        const float4 x0 = *reinterpret_cast<const float4*>(sm + OFF_XS + xs_off(r, ch0));
        const float4 x1 = *reinterpret_cast<const float4*>(sm + OFF_XS + xs_off(r, ch0 + 4));
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t o1[4], o2[4];
        float bk[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 vv = unpack_bf16(rw[e]);
          const int ca = ch0 + 2 * e, cb = ca + 1;
          float ha = vv.x * nrm, hb = vv.y * nrm;
          float kba = ha, kbb = hb;  // Kbar's k (never gated)
          if (CG && krole) {  // erase gate b = sigmoid(raw) on the row side of Abar and in W's operand
            const float2 ee = unpack_bf16(re[e]);
            ha *= sigmoid_fast(ee.x);
            hb *= sigmoid_fast(ee.y);
          }
          const float sa = ex2(xv[2 * e]), sbv = ex2(xv[2 * e + 1]);  // e^{G_r - B_{I+1}} >= 1
          const float ia = ex2(-xv[2 * e]), ib = ex2(-xv[2 * e + 1]);  // e^{B_{I+1} - G_r} <= 1
          rowf[8 * cc + 2 * e] = ha * sa;
          rowf[8 * cc + 2 * e + 1] = hb * sbv;
          const float ga = sa * s_eB[pI * 128 + ca], gb = sbv * s_eB[pI * 128 + cb];  // Gamma_r
          o1[e] = pack_h2(ha * ga, hb * gb);  // Kh*Gamma (k rows) or Qh*Gamma (q rows)
          if (krole) {
            o2[e] = pack_h2(kba * ia * s_eK[pI * 128 + ca], kbb * ib * s_eK[pI * 128 + cb]);  // Kbar
          } else {
            const float2 kk = unpack_bf16(rk[e]);
            bk[2 * e] = kk.x * nrmk * ia;  // kh_r e^{B_{I+1} - G_r}
            bk[2 * e + 1] = kk.y * nrmk * ib;
          }
        }
        if (krole) {
          *reinterpret_cast<uint4*>(sm + OFF_XW + sw128_chunk(r, 8 * hh + cc, 64)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<uint4*>(sm + OFF_B2A + sw128_chunk(r, 8 * hh + cc, 64)) =
              make_uint4(o2[0], o2[1], o2[2], o2[3]);
        } else {
          *reinterpret_cast<uint4*>(sm + OFF_B1 + sw128_chunk(64 + r, 8 * hh + cc, 128)) =
              make_uint4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<float4*>(sm + OFF_BK + sw128_off32(r, ch0, 64)) = make_float4(bk[0], bk[1], bk[2], bk[3]);
          *reinterpret_cast<float4*>(sm + OFF_BK + sw128_off32(r, ch0 + 4, 64)) = make_float4(bk[4], bk[5], bk[6], bk[7]);
        }
      }
    }
    fence_async_smem();
    KDA_SYNC_OR_BAIL();
    KDA_STAGE(FS_OPERANDS);
    // staged q, k, g and the decay offsets are consumed: fetch v of this
    // chunk (into the offsets' space) and q, k, g of the next chunk
    if (tid == 0) {
      issue_v(static_cast<int>(t0));
      const int cn = split ? c + 2 : c + 1;  // the next chunk this CTA prepares itself
      if (helper) {
        if (nx_c >= 0) issue_next_job();
      } else if (cn < nchunks) {
        issue_qkg(h, static_cast<int>(bos + static_cast<int64_t>(cn) * kC));
      }
    }

    // ---- Abar | M by column block J: tf32, row operand in TMEM. Rounds 0-2
    // are written at once and issued in parallel by lane 0 of warps 0-2 (each
    // commits to its own mbarrier); round 3 reuses round 0's columns. Rows of
    // blocks before J do not contribute to column block J (s > r), but every
    // lane stores: tcgen05.st is warp-collective. ----
    auto store_round = [&](int J, uint32_t aj) {
      float uv[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int ch = 64 * hh + 32 * half + j;
          const float u = (J < pI) ? s_u[(pI * (pI - 1) / 2 + J) * 128 + ch] : 1.f;
          uv[j] = rowf[32 * half + j] * u;
        }
        tmem_st32(tmem + tlane + aj + 64 * hh + 32 * half, uv);
      }
    };
    auto issue_round = [&](int J, uint32_t aj, uint64_t* done) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < 16; ++ks)
        mma_tf32_ta(tmem + TM_DA + 16 * J, tmem + aj + 8 * ks, desc_k(D0, OFF_BK, 64, 16 * J, ks),
                    idesc_tf32(128, 16), ks > 0);
      mma_commit(done);
    };
#pragma unroll 1
    for (int J = 0; J < 3; ++J) store_round(J, TM_AJ + 128 * J);
    tmem_st_wait();
    fence_before_sync();
    KDA_SYNC_OR_BAIL();
    if (lane == 0 && warp < 3) issue_round(warp, TM_AJ + 128 * warp, warp == 0 ? bar_mma : (warp == 1 ? bar_odd : bar_r2));
    KDA_WAIT(bar_mma, ph_mma);  // round 0 has read its columns
    fence_after_sync();
    store_round(3, TM_AJ);
    tmem_st_wait();
    fence_before_sync();
    KDA_SYNC_OR_BAIL();
    if (tid == 0) {
      issue_round(3, TM_AJ, bar_mma);
      if (pub_pending) publish();  // the previous job's stores have long completed
    }
    pub_pending = false;
    KDA_WAIT(bar_odd, ph_odd);  // round 1
    KDA_WAIT(bar_r2, ph_r2);    // round 2
    KDA_WAIT(bar_mma, ph_mma);  // round 3
    KDA_STAGE(FS_ROUNDS);
    fence_after_sync();

    // ---- Abar (fp32, for the inverse) and M (fp16 operand) out of TMEM ----
    {
      float v[32];
      tmem_ld32(tmem + tlane + TM_DA + 32 * hh, v);
      const int m = lrow;
      if (m < 64) {
        float* Ab = reinterpret_cast<float*>(sm + OFF_ABAR);  // diag(beta) Abar
        const float bm = s_beta[m];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int s = 32 * hh + j;
          Ab[m * 65 + s] = s < m ? bm * v[j] : 0.f;
        }
      } else {
        const int r = m - 64;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 32 * hh + 8 * cc + 2 * e;
            w[e] = pack_h2(s <= r ? v[8 * cc + 2 * e] : 0.f, s + 1 <= r ? v[8 * cc + 2 * e + 1] : 0.f);
          }
          *reinterpret_cast<uint4*>(sm + OFF_B2B + sw128_chunk(r, 4 * hh + cc, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    fence_before_sync();
    __syncthreads();
    KDA_STAGE(FS_ROUND_READOUT);
    tri_inverse(sm, s_beta, tid);
    KDA_STAGE(FS_INVERSE);
    if (CG) {  // T is consumed: the write gate takes its space
      __syncthreads();
      if (tid == 0) {
        mbar_expect_tx(bar_w, 2 * 8192);
        tma_load_3d(sm + OFF_WG, &tmw, 0, h, static_cast<int>(t0), bar_w);
        tma_load_3d(sm + OFF_WG + 8192, &tmw, 64, h, static_cast<int>(t0), bar_w);
      }
    }
    // ---- low part of M (its fp32 values are still in TMEM) ----
    {
      float v[32];
      tmem_ld32(tmem + tlane + TM_DA + 32 * hh, v);
      if (lrow >= 64) {
        const int r = lrow - 64;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 32 * hh + 8 * cc + 2 * e;
            const float m0 = s <= r ? v[8 * cc + 2 * e] : 0.f, m1 = s + 1 <= r ? v[8 * cc + 2 * e + 1] : 0.f;
            const uint32_t hi = pack_h2(m0, m1);
            const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            w[e] = pack_h2(m0 - hf.x, m1 - hf.y);
          }
          *reinterpret_cast<uint4*>(sm + OFF_ML + sw128_chunk(r, 4 * hh + cc, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    // ---- v (bf16, TMA) -> fp16 in place ----
    KDA_WAIT(bar_v, ph_v);
    if (CG) KDA_WAIT(bar_w, ph_w);
    {
      uint4* vt = reinterpret_cast<uint4*>(sm + OFF_V);
      const uint4* wt = reinterpret_cast<const uint4*>(sm + OFF_WG);  // same layout as v
#pragma unroll
      for (int x = tid; x < 16384 / 16; x += kThreads) {
        uint4 w = vt[x];
        float2 a0 = unpack_bf16(w.x), a1 = unpack_bf16(w.y), a2 = unpack_bf16(w.z), a3 = unpack_bf16(w.w);
        if (CG) {  // GDN-2: U = T (w * v), write gate w = sigmoid(raw)
          const uint4 ww = wt[x];
          const float2 w0 = unpack_bf16(ww.x), w1 = unpack_bf16(ww.y), w2 = unpack_bf16(ww.z), w3 = unpack_bf16(ww.w);
          a0.x *= sigmoid_fast(w0.x); a0.y *= sigmoid_fast(w0.y);
          a1.x *= sigmoid_fast(w1.x); a1.y *= sigmoid_fast(w1.y);
          a2.x *= sigmoid_fast(w2.x); a2.y *= sigmoid_fast(w2.y);
          a3.x *= sigmoid_fast(w3.x); a3.y *= sigmoid_fast(w3.y);
        }
        vt[x] = make_uint4(pack_h2(a0.x, a0.y), pack_h2(a1.x, a1.y), pack_h2(a2.x, a2.y), pack_h2(a3.x, a3.y));
      }
    }
    fence_async_smem();
    fence_before_sync();
    KDA_SYNC_OR_BAIL();
    if (tid == 0) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // W^T = (Kh Gamma)^T (T'hi + T'lo)^T
        mma(tmem + TM_DW, desc_mn(D0, OFF_XW, 8192, ks & 3),
            desc_k(D0, (ks < 4 ? OFF_TP : OFF_TPL), 64, 0, ks & 3), idesc(128, 64, true, false), ks > 0);
      if (!helper) issue_u();  // a helper hands v and T' over instead
      mma_commit(bar_mma);
    }
    KDA_WAIT(bar_mma, ph_mma);
    fence_after_sync();

    KDA_STAGE(FS_WU);
    // ---- -W into rows 0..63 of B1 ----
    {
      float v[32];
      tmem_ld32(tmem + tlane + TM_DW + 32 * hh, v);  // lane = channel i, columns r
#pragma unroll
      for (int j = 0; j < 32; ++j)
        *reinterpret_cast<__half*>(sm + OFF_B1 + sw128_off(32 * hh + j, lrow, 128)) = __float2half_rn(-v[j]);
    }
    fence_async_smem();
    fence_before_sync();
    KDA_SYNC_OR_BAIL();
    KDA_STAGE(FS_NEG_W);
    }  // prepared here
    if (helper) {
      // ---- hand the prepared odd chunk over: the operand runs, T' hi and
      // gamma to the item's slot once the main CTA has drained it; the stores
      // complete, and are published, during the next job ----
      if (tid == 0) {
        const int tt = c >> 1;
        if (tt >= kXSlots && !wait_flag_geq(a.xflags + 5 * item + 4, static_cast<uint32_t>(tt - kXSlots + 1), a.status))
          *s_fail = 1;
        fence_proxy_global();
        uint8_t* slot = a.xbuf + (static_cast<size_t>(item) * kXSlots + tt % kXSlots) * kXSlotBytes;
        bulk_store(slot + kXB, sb + OFF_B1, kXBBytes);
        bulk_store(slot + kXR, sb + OFF_V, kXRBytes);
        bulk_store(slot + kXTP, sb + OFF_TP, 8192);
        bulk_store(slot + kXGAM, smem_addr(s_gam), 512);
        pub_item = item;
        pub_tt = tt;
      }
      pub_pending = true;
      KDA_STAGE(FS_HANDOFF);
      continue;
    }
    if (handed) {
      // ---- a helper prepared this chunk; its operands landed during the
      // previous chunk, and the slot is free again ----
      if (mbar_wait(bar_x, ph_x, a.status, wait_limit))
        x_pending = false;
      else
        *s_fail = 1;
      ph_x ^= 1u;
      if (tid == 0) st_release(a.xflags + 5 * item + 4, static_cast<uint32_t>((c >> 1) + 1));
      KDA_STAGE(FS_SLOT_WAIT);
    }
    if (tid == 0) {
      fence_after_sync();
      if (handed) issue_u();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // U~^T = U^T + H^T (-W)^T
        mma(tmem + TM_DU, desc_k(D0, OFF_A1, 128, 0, ks), desc_k(D0, OFF_B1, 128, 0, ks), idesc(128, 64), 1);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // O^T = H^T (Qh Gamma)^T
        mma(tmem + TM_DO, desc_k(D0, OFF_A1, 128, 0, ks), desc_k(D0, OFF_B1, 128, 64, ks), idesc(128, 64),
            ks > 0);
      mma_commit(bar_mma);
    }
    KDA_WAIT(bar_mma, ph_mma);
    fence_after_sync();

    KDA_STAGE(FS_UT_O);
    // ---- U~^T (fp16) as the A operand of the Kbar and M products ----
    {
      float v[32];
      tmem_ld32(tmem + tlane + TM_DU + 32 * hh, v);  // lane = v, columns r
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float x0 = v[8 * cc + 2 * e], x1 = v[8 * cc + 2 * e + 1];
          hw[e] = pack_h2(x0, x1);
          const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hw[e]));
          lw[e] = pack_h2(x0 - hf.x, x1 - hf.y);
        }
        *reinterpret_cast<uint4*>(sm + OFF_XW + sw128_chunk(lrow, 4 * hh + cc, 128)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(sm + OFF_UL + sw128_chunk(lrow, 4 * hh + cc, 128)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    fence_async_smem();
    fence_before_sync();
    KDA_SYNC_OR_BAIL();
    if (tid == 0) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)  // (Kbar^T U~)^T = U~^T Kbar
        mma(tmem + TM_DH, desc_k(D0, OFF_XW, 128, 0, ks), desc_mn(D0, OFF_B2A, 8192, ks),
            idesc(128, 128, false, true), ks > 0);
#pragma unroll
      for (int ks = 0; ks < 12; ++ks) {  // O^T += U~hi^T Mhi^T + U~hi^T Mlo^T + U~lo^T Mhi^T
        const uint32_t ua = (ks < 8) ? OFF_XW : OFF_UL;
        const uint32_t mb = (ks >= 4 && ks < 8) ? OFF_ML : OFF_B2B;
        mma(tmem + TM_DO, desc_k(D0, ua, 128, 0, ks & 3), desc_k(D0, mb, 64, 0, ks & 3), idesc(128, 64), 1);
      }
      mma_commit(bar_mma);
    }
    KDA_WAIT(bar_mma, ph_mma);
    fence_after_sync();
    KDA_STAGE(FS_KBAR_M);
    if (split && !(c & 1) && c + 1 < nchunks) {
      // fetch the helper-prepared next (odd) chunk into the tiles this chunk
      // has finished with (its last product above has completed)
      if (tid == 0) {
        const int tt = (c + 1) >> 1;
        if (!wait_flag_geq(a.xflags + 5 * item + tt % kXSlots, static_cast<uint32_t>(tt + 1), a.status)) *s_fail = 1;
        fence_proxy_global();
        const uint8_t* slot = a.xbuf + (static_cast<size_t>(item) * kXSlots + tt % kXSlots) * kXSlotBytes;
        mbar_expect_tx(bar_x, kXSlotBytes);
        bulk_load(sb + OFF_B1, slot + kXB, kXBBytes, bar_x);
        bulk_load(sb + OFF_V, slot + kXR, kXRBytes, bar_x);
        bulk_load(sb + OFF_TP, slot + kXTP, 8192, bar_x);
        bulk_load(smem_addr(s_gam2), slot + kXGAM, 512, bar_x);
      }
      x_pending = true;
    }

    KDA_STAGE(FS_NEXT_SLOT);
    // ---- state update (fp32 registers), next H^T operand, output ----
    {
      float v[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld32(tmem + tlane + TM_DH + 64 * hh + 32 * half, v);
        const float4* g4 = reinterpret_cast<const float4*>((handed ? s_gam2 : s_gam) + 64 * hh + 32 * half);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 gm = g4[j4];
          const int j = 32 * half + 4 * j4;
          Hst[j] = gm.x * Hst[j] + v[4 * j4];
          Hst[j + 1] = gm.y * Hst[j + 1] + v[4 * j4 + 1];
          Hst[j + 2] = gm.z * Hst[j + 2] + v[4 * j4 + 2];
          Hst[j + 3] = gm.w * Hst[j + 3] + v[4 * j4 + 3];
        }
      }
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(sm + OFF_A1 + sw128_chunk(lrow, 8 * hh + cc, 128)) =
            make_uint4(pack_h2(Hst[8 * cc], Hst[8 * cc + 1]), pack_h2(Hst[8 * cc + 2], Hst[8 * cc + 3]),
                       pack_h2(Hst[8 * cc + 4], Hst[8 * cc + 5]), pack_h2(Hst[8 * cc + 6], Hst[8 * cc + 7]));
      tmem_ld32(tmem + tlane + TM_DO + 32 * hh, v);  // lane = v, columns r
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int r = 32 * hh + j;
        if (r < rows) a.o[((t0 + r) * a.H + h) * kD + lrow] = __float2bfloat16_rn(v[j]);
      }
    }
    fence_async_smem();
    fence_before_sync();
    KDA_SYNC_OR_BAIL();
  }
  if (!helper && a.hT != nullptr) {  // final state
    float* dst = a.hT + static_cast<int64_t>(item) * (kD * kD);
#pragma unroll
    for (int j = 0; j < 64; ++j) dst[(64 * hh + j) * kD + lrow] = Hst[j];
  }
#undef KDA_WAIT
#undef KDA_SYNC_OR_BAIL
teardown:
  // no async copy may still target this CTA's shared memory when it exits
  if (x_pending) mbar_wait(bar_x, ph_x, a.status, wait_limit);
  if (tid == 0) {
    if (pub_pending)
      publish();
    else
      bulk_wait_all();
  }
  fence_before_sync();
  __syncthreads();
  KDA_STAGE_FLUSH(g_fwd_stage);
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

// [S][H][128] bf16 tensor, box = 64 channels x 1 head x 64 tokens, 128-byte swizzle.
bool make_tma_map_bf16(CUtensorMap* m, const void* base, int64_t S, int H) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(H) * kD * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t fwd_handoff_bytes(int items) {
  const size_t flags = (static_cast<size_t>(items) * 5 * sizeof(uint32_t) + 255) / 256 * 256;
  return flags + static_cast<size_t>(items) * kXSlots * kXSlotBytes;
}

kda_status launch_fwd_tc(const kda_problem* p, const FwdArgs& a, cudaStream_t s) {
  if (p->head_dim != kD || p->dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;
  const bool cg = a.w != nullptr;  // GDN-2: b is the raw erase gate [S,H,D], w the raw write gate
  CUtensorMap mq, mk, mv, mg, me, mw;
  if (!make_tma_map_bf16(&mq, a.q, p->total_tokens, p->num_heads) ||
      !make_tma_map_bf16(&mk, a.k, p->total_tokens, p->num_heads) ||
      !make_tma_map_bf16(&mv, a.v, p->total_tokens, p->num_heads) ||
      !make_tma_map_bf16(&mg, a.g, p->total_tokens, p->num_heads))
    return KDA_ERR_CUDA;
  if (cg) {
    if (!make_tma_map_bf16(&me, a.b, p->total_tokens, p->num_heads) ||
        !make_tma_map_bf16(&mw, a.w, p->total_tokens, p->num_heads))
      return KDA_ERR_CUDA;
  } else {
    me = mq;  // unused
    mw = mq;
  }
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const CUtensorMap, const TcFwdArgs) = cg ? kda_fwd_tc_kernel<true> : kda_fwd_tc_kernel<false>;
  TcFwdArgs t;
  t.b = static_cast<const __nv_bfloat16*>(a.b);
  t.A_log = a.A_log;
  t.dt_bias = a.dt_bias;
  t.o = static_cast<__nv_bfloat16*>(a.o);
  t.h0 = a.h0;
  t.hT = a.hT;
  t.ckpt = a.ckpt;
  t.status = a.status;
  t.cu = a.cu;
  t.S = a.S;
  t.N = a.N;
  t.H = a.H;
  t.scale = a.scale;
  t.lower = a.lower;
  t.eps = a.eps;
  t.test_timeout = a.test_timeout;
  t.helpers = 0;
  t.xflags = a.xflags;
  t.xbuf = a.xbuf;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
    return KDA_ERR_CUDA;
  const int items = p->num_seqs * p->num_heads;
  // Split mode: with at least half as many spare SMs as items, helper CTAs
  // prepare every other chunk. Their hand-off waits need every CTA resident
  // at once, which a cooperative launch guarantees (or refuses, and the
  // plain launch runs instead).
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, SMEM_BYTES);
  bool launched = false;
  if (a.xflags != nullptr && !a.test_timeout && items > 0 && items < sms * per_sm) {
    const int spare = sms * per_sm - items;
    if (2 * spare >= items) {
      t.helpers = spare < items ? spare : items;
      if (cudaMemsetAsync(a.xflags, 0, sizeof(uint32_t) * 5 * items, s) != cudaSuccess) return KDA_ERR_CUDA;
      void* kargs[] = {&mq, &mk, &mv, &mg, &me, &mw, &t};
      launched = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern),
                                             dim3(items + t.helpers), dim3(kThreads), kargs, SMEM_BYTES,
                                             s) == cudaSuccess;
      if (!launched) {
        cudaGetLastError();  // clear the refusal; run without helpers
        t.helpers = 0;
      }
    }
  }
  if (!launched && items > 0) kern<<<items, kThreads, SMEM_BYTES, s>>>(mq, mk, mv, mg, me, mw, t);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
