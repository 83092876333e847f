// kda_tc_bwd.cu -- tensor-core KDA backward (bf16 inputs, D = K = V = 128) with
// the recompute policy: the forward keeps one fp32 state per 1024 tokens; per
// such segment (walked in reverse) the backward rebuilds the chunk-start
// states, keeps them as fp16 tiles in per-CTA scratch, then walks the
// segment's chunks in reverse, recomputing each chunk's WY factors and gated
// q/k from the inputs and propagating the state gradient dH.
//
// Chunk size C = 16: every factor exp(+-(G_r - G_s)) inside a chunk then stays
// within fp32 range ("KDA at the production shape ...", section 3(a): the
// inverse-decay factor of k leaves fp32 range once the cumulative log-decay
// passes -88, i.e. beyond 17 tokens at the -5 floor). Work split:
//   * state products (128-long contractions or 128 x 128 results): tcgen05,
//     fp16 operands, fp32 accumulators in TMEM (lanes = value index v or key
//     index i); both fp32 states live in TMEM (H^T while rebuilding, dH^T);
//   * the 16 x 16 intra-chunk matrices, the WY factors and every gradient
//     product with a 16-long contraction: warp-level tf32 tensor-core tiles
//     (mma.sync m16n8k8; tcgen05's smallest tile has 64 rows), with operands
//     split into tf32 hi + lo parts so the products keep fp32 accuracy;
//   * gate / cumulative-sum / L2-norm elementwise work: CUDA cores.
// Each chunk's q/k/v/g (and dO) tiles are prefetched one chunk ahead with
// async copies; the fp16 chunk-start states move to and from scratch with
// bulk async copies.
//
// Per chunk (r, s in 0..15; G chunk-local cumulative log-decay; Gamma = e^G;
// T' = T diag(beta), T = (I + diag(beta) Abar)^-1):
//   U~ = T' V - T' (Kh Gamma) H          O-side:  dQG = dO H^T,  dM = dO U~^T
//   dU~ = M^T dO + Kbar dH'               dH = diag(gamma) dH' + (Qh Gamma)^T dO - W^T dU~
//   dW = -dU~ H^T,  dKbar = U~ dH'^T,  dgamma = rowsum(H .* dH')
//   dT' = dW (Kh Gamma)^T + dU~ V^T,  dV = T'^T dU~,  d(Kh Gamma) += T'^T dW
//   dA = -T^T (dT' diag(beta)) T^T,  then Abar / M / gate / L2-norm chain rules.
#include "kda_tc_common.cuh"

#ifdef KDA_STAGE_TIMERS
// per-CTA stage counters of the tensor-core backward (tracing build)
__device__ unsigned long long g_bwd_stage[kStageCtas * 32];
extern "C" int kda_bwd_stage_timers(unsigned long long* host, int clear) {
  static unsigned long long zero[kStageCtas * 32];
  if (host != nullptr && cudaMemcpyFromSymbol(host, g_bwd_stage, sizeof(g_bwd_stage)) != cudaSuccess) return 1;
  if (clear && cudaMemcpyToSymbol(g_bwd_stage, zero, sizeof(zero)) != cudaSuccess) return 1;
  return 0;
}
#endif

namespace kda {
namespace {
using namespace tc;

constexpr int kC = 16;
constexpr int kD = 128;
constexpr int kT = 256;
constexpr int kCPS = kCkptTokens / kC;  // chunks per checkpoint segment (64)
constexpr int kLd = 132;                // fp32 tile row stride (floats)
constexpr int kTileF = kC * kLd * 4;    // bytes of one fp32 [16][132] tile
constexpr int kSq = 20;                 // row stride of the 16 x 16 matrices
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kStateBytes = 32768;  // fp16 128 x 128 state tile
// One scratch slot per chunk: the chunk-start state and, in split mode, what
// a helper CTA prepares for the reverse CTA: the chunk's Abar, T, T' (the
// 16 x kSq small matrices at S_AB .. S_TP), the M hi / lo tiles, -W and U~
// (fp16 operand tiles) and U~ (fp32 tile).
constexpr uint32_t kPrepSBytes = 3 * 320 * 4;  // S_AB, S_T, S_TP
constexpr uint32_t kPrepMBytes = 4096;         // M hi + lo tiles
constexpr uint32_t kPrepWOff = kStateBytes + 8192;  // -W fp16 [16][128]
constexpr uint32_t kPrepUOff = kPrepWOff + 4096;    // U~ fp16 [16][128]
constexpr uint32_t kPrepUTOff = kPrepUOff + 4096;   // U~ fp32 [16][kLd]
constexpr uint32_t kSlotBytesSplit = kPrepUTOff + kC * kLd * 4;
constexpr uint32_t kSlotBytesInline = kStateBytes;  // the state alone
// The first and the last chunk of a sequence also keep the fp16 low part of
// their start state (the state minus its fp16 value) in a per-item edge
// area of the workspace (two 32 KB tiles per (sequence, head)): there the
// state or the state gradient is the caller's (h0, dhT), and the gate
// gradient of the chunk's tokens is dominated by dgamma = rowsum(H .* dH'),
// a direct product of the two, which then needs the state to better than
// fp16 (~2^-22 with hi + lo). Inside a sequence both factors are the
// recurrence's own and the fp16 state meets the bar.
constexpr uint32_t kEdgeBytes = 2 * kStateBytes;

// Stages of a chunk step, as the stage timers of a tracing build count them
// (each mark closes the stage named by it).
enum BwdStage {
  BS_JOB,           // a helper claims a job
  BS_HANDOFF,       // split mode: wait for a rebuilt segment / a free buffer
  BS_CKPT,          // segment start state from its checkpoint
  BS_TILES_ISSUE,   // the next chunk's q / k / v / g copies issued
  BS_STATE_STORE,   // rebuild pass: the chunk-start state's bulk store issued
  BS_TILES_WAIT,    // this chunk's tiles landed
  BS_TOP_BARRIER,   // barrier at the top of the step
  BS_NORM_GATE,     // row norms, gate, per-half cumulative sums
  BS_OPERANDS,      // full cumulative sum, gated operand tiles
  BS_SLOT_WAIT,     // split mode: the helper's matrices landed
  BS_DO_ISSUE,      // reverse pass: the next chunk's dO copies issued
  BS_ABAR_M,        // Abar / M tf32 tiles (and the dU~ MMA issue)
  BS_INVERSE,       // T = (I + diag(beta) Abar)^-1
  BS_WU,            // W, U
  BS_UT_MMA,        // U~ = U - W H (tcgen05) completed
  BS_DUT_MMA,       // dU~ (tcgen05) completed
  BS_READOUT,       // U~ / dU~ out of TMEM
  BS_REBUILD_MMA,   // rebuild pass: Kbar^T U~ (tcgen05) completed
  BS_STATE_UPDATE,  // rebuild pass: H <- diag(gamma) H + Kbar^T U~
  BS_DM,            // state MMAs issued; dM and dU~ V^T tiles
  BS_STATE_MMA,     // state MMAs completed
  BS_E,             // [E] dH update, dgamma, dQG / dW / dKbar readout
  BS_D1,            // [D1]
  BS_D2,            // [D2]
  BS_F,             // [F]
  BS_DG_CUMSUM,     // dG reverse cumulative sum
  BS_NORM_DOTS,     // L2-norm chain rule row dots
  BS_OUTPUTS,       // dq, dk, dg, dbeta out
  BS_COUNT
};
static_assert(BS_COUNT <= 31, "stage slots");

// ---- shared memory map (bytes) ----
constexpr int OFF_A1 = 0;                  // H^T fp16 [128 v][128 i] (SW128)
constexpr int OFF_A1D = 32768;             // dH'^T fp16 [128 v][128 i]
constexpr int OFF_FW = 65536;              // -W     fp16 [16 r][128 i]
constexpr int OFF_FQG = OFF_FW + 4096;     // Qh*Gamma fp16 [16 r][128 i]
constexpr int OFF_FKB = OFF_FQG + 4096;    // Kbar   fp16 [16 r][128 i]
constexpr int OFF_FDO = OFF_FKB + 4096;    // dO     fp16 [16 r][128 v]
constexpr int OFF_FU = OFF_FDO + 4096;     // U~     fp16 [16 r][128 v]
constexpr int OFF_FDU = OFF_FU + 4096;     // dU~    fp16 [16 r][128 v]
constexpr int OFF_FM = OFF_FDU + 4096;     // M hi (K-major B of dU~^T: row s, column r)
constexpr int OFF_FML = OFF_FM + 2048;     // M lo
constexpr int OFF_STG = OFF_FML + 2048;    // two buffers of q, k, v, g bf16 [16][128]
constexpr int kStgBuf = 4 * 4096;
constexpr int OFF_SDO = OFF_STG + 2 * kStgBuf;  // dO bf16 [16][128]
constexpr int OFF_F32 = OFF_SDO + 4096;         // fp32 [16][132] tiles
enum { T_GS = 0, T_QG, T_KG, T_KI, T_U, T_DU, T_W, T_AQ, T_AK, T_AG, NT32 };
constexpr int OFF_SMALL = OFF_F32 + NT32 * kTileF;
// small fp32 arrays (offsets in floats); 16 x 16 matrices with row stride kSq
constexpr int S_AB = 0, S_T = 320, S_TP = 640, S_DM = 960, S_DT1 = 1280, S_DT2 = 1600, S_Y = 1920, S_DAB = 2240;
constexpr int S_BETA = 2560, S_IQ0 = 2576, S_IK0 = 2592, S_DB = 2608, S_RQ = 2624, S_RK = 2640;
constexpr int S_GEND = 2656, S_DGE = 2784, S_TOT = 2912, S_PART = 3168, S_GAM = 3424, S_PR = 3552;
constexpr int SMALL_FLOATS = 3872;
constexpr int OFF_BAR = OFF_SMALL + SMALL_FLOATS * 4;
constexpr int OFF_STAGE = OFF_BAR + 64;  // stage counters (tracing build only)
constexpr int SMEM_BYTES = OFF_STAGE + KDA_STAGE_BYTES + 1024;  // + alignment slack
// The dgamma reduce-scatter lands in the M hi / lo tiles (free by then).
constexpr int OFF_RED = OFF_FM;
static_assert(OFF_STG % 1024 == 0 && OFF_F32 % 16 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

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
  const float* dhT;  // gradient of the final states [N][H][D][D] (NULL: zero)
  float* dh0;        // gradient of the initial states (NULL: not written)
  __nv_bfloat16 *dq, *dk, *dv, *dg, *db;
  float* partial;
  uint8_t* scratch;  // fp16 chunk-start state tiles (per CTA, or per item and level parity)
  uint8_t* edge;     // per item: low parts of the first and last chunk's start states
  uint32_t* flags;   // per item: last level + 1 rebuilt into each buffer, levels consumed (split mode)
  int* status;
  const int32_t* cu;
  int64_t S;  // total tokens (cu[N])
  int N, H;
  int helpers;  // > 0: CTAs N*H .. N*H+helpers-1 rebuild segment states for the others
  float scale, lower, eps;
  // forward with 16-token chunks (kFwd): output, initial / final states
  __nv_bfloat16* o;
  const float* h0;   // [N][H][D][D] (NULL: zero)
  float* hT;         // (NULL: not written)
  float* ckpt_out;   // checkpoints written (NULL: inference, none)
};

__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + ex2(-x * kLog2e)); }
__device__ __forceinline__ void st_h(uint8_t* base, uint32_t off, float x) {
  *reinterpret_cast<__half*>(base + off) = __float2half_rn(x);
}
__device__ __forceinline__ void st_h2(uint8_t* base, uint32_t off, float x0, float x1) {
  *reinterpret_cast<uint32_t*>(base + off) = pack_h2(x0, x1);
}
__device__ __forceinline__ float lo_part(float x) { return x - __half2float(__float2half_rn(x)); }
// element (r, c) of a bf16 [16][128] staging tile
__device__ __forceinline__ float stg(const uint8_t* tile, int r, int c) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + r * 256 + c * 2));
}
__device__ __forceinline__ float h16(const uint8_t* base, uint32_t off) {
  return __half2float(*reinterpret_cast<const __half*>(base + off));
}

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

// Async copies of the tiles of tokens [t0, t0 + 16) of head h into bf16
// [16][128] staging tiles (q, k, v, g at dst + 0/4/8/12 KB; dO at dst_dO);
// rows at or past `rows` are zero-filled. Every thread copies 16 bytes per tile.
__device__ __forceinline__ void stage_tiles(const TcBwdArgs& a, uint32_t dst, int h, int64_t t0, int rows, int tid,
                                            bool qkvg, bool dO, uint32_t dst_dO, bool with_q = true) {
  const int r = tid >> 4, j = tid & 15;
  const bool ok = r < rows;
  const int64_t off = ok ? ((t0 + r) * a.H + h) * kD + 8 * j : 0;
  const int n = ok ? 16 : 0;
  const uint32_t so = static_cast<uint32_t>(r * 256 + 16 * j);
  if (qkvg) {
    if (with_q) cp_async16(dst + 0 * 4096 + so, a.q + off, n);
    cp_async16(dst + 1 * 4096 + so, a.k + off, n);
    cp_async16(dst + 2 * 4096 + so, a.v + off, n);
    cp_async16(dst + 3 * 4096 + so, a.g + off, n);
  }
  if (dO) cp_async16(dst_dO + so, a.dO + off, n);
}

// Low part (value minus its fp16 rounding) of lane L's 64 state values
// (columns 64 hh ..) into an SW128 edge tile, from an fp32 [i][v] state in
// global memory (a checkpoint) or from the TMEM state (lane L, 64 columns at
// taddr). Out of line: they run once per sequence edge and must not weigh
// on the hot loop's registers.
__device__ __forceinline__ void lo_tile_store(uint8_t* tile, int L, int hh, int half, const float* x) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = x[8 * cc + 2 * e], x1 = x[8 * cc + 2 * e + 1];
      const uint32_t hi = pack_h2(x0, x1);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      w[e] = pack_h2(x0 - hf.x, x1 - hf.y);
    }
    *reinterpret_cast<uint4*>(tile + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
__device__ __noinline__ void edge_lo_from_global(uint8_t* tile, const float* src, int L, int hh) {
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = src[(64 * hh + 32 * half + j) * kD + L];
    lo_tile_store(tile, L, hh, half, x);
  }
}
__device__ __noinline__ void edge_lo_from_tmem(uint8_t* tile, uint32_t taddr, int L, int hh) {
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    float x[32];
    tmem_ld32(taddr + 32 * half, x);
    lo_tile_store(tile, L, hh, half, x);
  }
}
// RED[0..511] += RED[512..1023] (the edge chunk's low-part dgamma partials)
__device__ __noinline__ void edge_fold(float* red) {
  for (int x = static_cast<int>(threadIdx.x); x < 512; x += static_cast<int>(blockDim.x)) red[x] += red[512 + x];
}

// dgamma's low-part term of a sequence-edge chunk, sum_v Hlo[i][v] dH'[i][v]:
// thread (lane L, column half hh) multiplies the fp16 low part of the chunk's
// start state (edge tile `lo`, read past L1) with dH' (TMEM, columns of
// `dh_tmem`), reduces the 64 products over the warp's lanes and writes its
// two totals to red[base], red[base + 1]. Kept out of line: it runs for two
// chunks per sequence and must not weigh on the hot loop's registers.
__device__ __noinline__ void edge_dgamma_lo(const uint8_t* lo, uint32_t dh_tmem, int L, int hh, int lane, float* red) {
  float p[64];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float dh[32];
    tmem_ld32(dh_tmem + 32 * half, dh);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint4 lw = __ldcg(reinterpret_cast<const uint4*>(lo + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)));
      const uint32_t lu[4] = {lw.x, lw.y, lw.z, lw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 lf = __half22float2(*reinterpret_cast<const __half2*>(&lu[e]));
        p[32 * half + 8 * cc + 2 * e] = lf.x * dh[8 * cc + 2 * e];
        p[32 * half + 8 * cc + 2 * e + 1] = lf.y * dh[8 * cc + 2 * e + 1];
      }
    }
  }
  warp_reduce_scatter64(p, lane);
  const int base = 32 * ((lane >> 4) & 1) + 16 * ((lane >> 3) & 1) + 8 * ((lane >> 2) & 1) + 4 * ((lane >> 1) & 1) +
                   2 * (lane & 1);
  red[base] = p[0];
  red[base + 1] = p[1];
}

// kEdge: the caller passes dhT or asks for dh0 (states in play), so the
// first and last chunk of each sequence take dgamma's low-part term (the
// instantiation without it is the stateless path, free of that code).
// kFwd: the forward with 16-token chunks. Each CTA walks its items' chunks in
// order from h0 with the rebuild pass's stages, and per chunk also forms
// O = (Qh Gamma) H + M U~ (the first product on tcgen05 beside the state
// update, the second with 3xTF32 warp tiles) and, at every checkpoint
// boundary, stores the chunk-start state.
template <bool kEdge, bool kFwd>
__global__ void __launch_bounds__(kT, 1) kda_bwd_tc_kernel(const TcBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_addr(sm);
  const uint64_t D0 = sdesc(sb, 0);  // base of every tcgen05 shared-memory descriptor
  float* F = reinterpret_cast<float*>(sm + OFF_F32);
  float* GS = F + T_GS * (kTileF / 4);
  float* QG = F + T_QG * (kTileF / 4);
  float* KG = F + T_KG * (kTileF / 4);
  float* KI = F + T_KI * (kTileF / 4);
  float* UT = F + T_U * (kTileF / 4);
  float* DUT = F + T_DU * (kTileF / 4);
  float* WT = F + T_W * (kTileF / 4);
  float* AQ = F + T_AQ * (kTileF / 4);
  float* AK = F + T_AK * (kTileF / 4);
  float* AG = F + T_AG * (kTileF / 4);
  float* S = reinterpret_cast<float*>(sm + OFF_SMALL);
  float* RED = reinterpret_cast<float*>(sm + OFF_RED);
  const uint8_t* SDO = sm + OFF_SDO;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_a1 = bar + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 2);
  int* s_fail = reinterpret_cast<int*>(bar + 3);
  int* s_job = s_fail + 1;     // split mode: a helper's claimed job
  uint64_t* bar_du = bar + 4;  // dU~ products (issued early, reverse pass)
  uint64_t* bar_g1 = bar + 5;  // (H dU~^T) products
  uint64_t* bar_g2 = bar + 6;  // (dH' U~^T) products
  uint64_t* bar_sm = bar + 7;  // split mode: a chunk's Abar, T, T', M loaded from scratch

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ci = tid & 127, rh = tid >> 7;  // channel role: channel ci, rows 8*rh .. 8*rh+7
  const int q4 = warp & 3, hh = warp >> 2, L = 32 * q4 + lane;  // TMEM lane role
  const uint32_t tlane = static_cast<uint32_t>(32 * q4) << 16;
  const int fg = lane >> 2, ft = lane & 3;  // mma fragment role
  const float Lg = a.lower * kLog2e;

  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar_a1, 1);
    mbar_init(bar_du, 1);
    mbar_init(bar_g1, 1);
    mbar_init(bar_g2, 1);
    mbar_init(bar_sm, 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(s_tmem, TM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *s_tmem;
  KDA_STAGE_INIT(sm + OFF_STAGE);
  uint32_t ph = 0, ph_a1 = 0, ph_du = 0, ph_g1 = 0, ph_g2 = 0, ph_sm = 0;
  bool sm_pending = false;  // a bulk load of a chunk's small matrices is in flight
  bool a1_pending = false;  // a bulk load into A1 is in flight (same value in every thread)
  // split mode, thread 0: a chunk's helper-prepared operands, scratch slot <-> shared memory
  auto load_prep = [&](const uint8_t* slot) {
    mbar_expect_tx(bar_sm, kPrepSBytes + kPrepMBytes + 8192 + kTileF);
    bulk_load(sb + OFF_SMALL, slot + kStateBytes, kPrepSBytes, bar_sm);
    bulk_load(sb + OFF_FM, slot + kStateBytes + kPrepSBytes, kPrepMBytes, bar_sm);
    bulk_load(sb + OFF_FW, slot + kPrepWOff, 4096, bar_sm);
    bulk_load(sb + OFF_FU, slot + kPrepUOff, 4096, bar_sm);
    bulk_load(sb + OFF_F32 + T_U * kTileF, slot + kPrepUTOff, kTileF, bar_sm);
  };
  auto ship_wu = [&](uint8_t* slot) {
    bulk_store(slot + kPrepWOff, sb + OFF_FW, 4096);
    bulk_store(slot + kPrepUOff, sb + OFF_FU, 4096);
    bulk_store(slot + kPrepUTOff, sb + OFF_F32 + T_U * kTileF, kTileF);
  };

#define KDA_WAIT_MMA()                              \
  do {                                              \
    if (!mbar_wait(bar, ph, a.status)) *s_fail = 1; \
    ph ^= 1u;                                       \
  } while (0)
#define KDA_SYNC_OR_BAIL()      \
  do {                          \
    __syncthreads();            \
    if (*s_fail) goto teardown; \
  } while (0)

  // Work iteration. A reverse CTA walks its items (blockIdx.x, + gridDim.x,
  // ...) and each item's segments from the last. In split mode (helpers > 0,
  // one reverse CTA per item) the helper CTAs rebuild the segment states:
  // the jobs (level L = segment nseg-1-L, item) are numbered level-major,
  // job = L * items + item, and a free helper claims the next one from a
  // global counter, so the levels complete in order, ahead of the reverse
  // CTAs; each item has kTcBwdBufs scratch buffers.
  const int items = a.N * a.H;
  const bool split = a.helpers > 0;
  const bool helper = split && static_cast<int>(blockIdx.x) >= items;
  int item = helper ? 0 : static_cast<int>(blockIdx.x);
  int seg = -1, lvl = 0;
  bool open = false;
  int max_jobs = 0;
  if (helper) {  // jobs run up to the longest sequence's segment count
    int max_seg = 0;
    for (int s2 = 0; s2 < a.N; ++s2)
      max_seg = max(max_seg, static_cast<int>((a.cu[s2 + 1] - a.cu[s2] + kCkptTokens - 1) / kCkptTokens));
    max_jobs = max_seg * items;
  }
  int n = 0, h = 0, nchunks = 0, nseg = 0;
  int64_t bos = 0, eos = 0;
  float expA = 0.f, dtb = 0.f, acc_dtb = 0.f, acc_alog = 0.f;

  while (true) {
    if (!helper) {
      if (!open) {
        if (item >= items) break;
        n = item / a.H;
        h = item % a.H;
        bos = a.cu[n];
        eos = a.cu[n + 1];
        nchunks = static_cast<int>((eos - bos + kC - 1) / kC);
        nseg = static_cast<int>((eos - bos + kCkptTokens - 1) / kCkptTokens);
        expA = expf(a.A_log[h]);
        dtb = a.dt_bias[h * kD + ci];
        acc_dtb = 0.f;
        acc_alog = 0.f;
        open = true;
        seg = kFwd ? 0 : nseg - 1;
        // dH' = dhT, the gradient of the final state, or zero (TMEM state and its
        // fp16 operand copy; lane = value channel L, columns = key channel); the
        // forward starts H from h0 or zero instead
        if constexpr (kFwd) {
          const float* src = a.h0 != nullptr ? a.h0 + static_cast<int64_t>(item) * (kD * kD) : nullptr;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = src != nullptr ? src[(64 * hh + 32 * half + j) * kD + L] : 0.f;
            tmem_st32(tmem + tlane + TM_H + 64 * hh + 32 * half, x);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(sm + OFF_A1 + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)) =
                  make_uint4(pack_h2(x[8 * cc], x[8 * cc + 1]), pack_h2(x[8 * cc + 2], x[8 * cc + 3]),
                             pack_h2(x[8 * cc + 4], x[8 * cc + 5]), pack_h2(x[8 * cc + 6], x[8 * cc + 7]));
          }
          tmem_st_wait();
        } else if (a.dhT != nullptr) {
          const float* src = a.dhT + static_cast<int64_t>(item) * (kD * kD);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = src[(64 * hh + 32 * half + j) * kD + L];
            tmem_st32(tmem + tlane + TM_DH + 64 * hh + 32 * half, x);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              *reinterpret_cast<uint4*>(sm + OFF_A1D + sw128_chunk(L, 8 * hh + 4 * half + cc, 128)) =
                  make_uint4(pack_h2(x[8 * cc], x[8 * cc + 1]), pack_h2(x[8 * cc + 2], x[8 * cc + 3]),
                             pack_h2(x[8 * cc + 4], x[8 * cc + 5]), pack_h2(x[8 * cc + 6], x[8 * cc + 7]));
          }
          tmem_st_wait();
        } else {
          float z[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = 0.f;
          tmem_st32(tmem + tlane + TM_DH + 64 * hh, z);
          tmem_st32(tmem + tlane + TM_DH + 64 * hh + 32, z);
          tmem_st_wait();
          for (int x = tid; x < 32768 / 16; x += kT) reinterpret_cast<uint4*>(sm + OFF_A1D)[x] = make_uint4(0, 0, 0, 0);
        }
      }
    } else {
      // claim the next job (a counter after the items' hand-off counters): a
      // helper blocked on one item's buffer holds back no other item's job
      bool found = false;
      while (true) {
        if (tid == 0) *s_job = static_cast<int>(atomicAdd(a.flags + kTcBwdFlags * items, 1u));
        KDA_STAGE(BS_JOB);
        __syncthreads();
        const int jb = *s_job;
        __syncthreads();
        if (jb >= max_jobs) break;
        lvl = jb / items;
        item = jb % items;
        n = item / a.H;
        h = item % a.H;
        bos = a.cu[n];
        eos = a.cu[n + 1];
        nchunks = static_cast<int>((eos - bos + kC - 1) / kC);
        nseg = static_cast<int>((eos - bos + kCkptTokens - 1) / kCkptTokens);
        if (lvl < nseg) {
          found = true;
          break;
        }
      }
      if (!found) break;
      seg = nseg - 1 - lvl;
      expA = expf(a.A_log[h]);
      dtb = a.dt_bias[h * kD + ci];
    }

    if (seg >= 0) {
      const int lv = nseg - 1 - seg;  // level: segments counted from the end
      // (the forward walks the whole sequence as one stretch)
      const int c0 = kFwd ? 0 : seg * kCPS, c1 = kFwd ? nchunks : min(nchunks, c0 + kCPS);
      const bool rebuild = !split || helper;
      const uint32_t sbytes = split ? kSlotBytesSplit : kSlotBytesInline;
      // edge tile of chunk c (0: the sequence's first chunk, 1: its last)
      uint8_t* edge_buf = a.edge + static_cast<size_t>(item) * kEdgeBytes;
      uint8_t* segbuf = split ? a.scratch + (static_cast<size_t>(item) * kTcBwdBufs + lv % kTcBwdBufs) * kCPS * sbytes
                              : a.scratch + static_cast<size_t>(blockIdx.x) * kCPS * sbytes;
      if (split) {  // hand-off: the helper waits until the level that last used this
                    // buffer (lv - kTcBwdBufs) is consumed, the reverse CTA until level lv is rebuilt
        if (tid == 0) {
          bool ok = true;
          uint32_t* f = a.flags + kTcBwdFlags * item;
          if (helper && lv >= kTcBwdBufs)
            ok = wait_flag_geq(f + kTcBwdBufs, static_cast<uint32_t>(lv - kTcBwdBufs + 1), a.status);
          if (!helper) ok = wait_flag_geq(f + lv % kTcBwdBufs, static_cast<uint32_t>(lv + 1), a.status);
          if (!ok) *s_fail = 1;
          fence_proxy_global();
        }
        KDA_SYNC_OR_BAIL();
        KDA_STAGE(BS_HANDOFF);
      }
      if constexpr (!kFwd) {  // (the forward starts from h0, set up at the item's start)
        if (rebuild) {
          // ---- segment start state: checkpoint (fp32 [i][v]) -> TMEM H^T and fp16 A1 ----
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
          if (kEdge && (c0 == 0 || c0 == nchunks - 1))  // a sequence-edge chunk starts at this checkpoint
            edge_lo_from_global(edge_buf + (c0 == 0 ? 0 : kStateBytes), src, L, hh);
          KDA_STAGE(BS_CKPT);
          fence_async_smem();
          fence_before_sync();
          __syncthreads();
        }
      }
      if constexpr (kFwd) {  // the state set up at the item's start feeds the first chunk's MMAs
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
      }

      // Pass 0 rebuilds the chunk-start states c0+1 .. c1-1 (state c is saved
      // to scratch slot c - c0 before chunk c advances it); pass 1 walks the
      // chunks c1-1 .. c0 in reverse.
#pragma unroll 1
      for (int pass = rebuild ? 0 : 1; pass < ((helper || kFwd) ? 1 : 2); ++pass) {
        const bool rev = pass == 1;
        // a helper also walks the segment's last chunk (its Abar, T, T', M only);
        // the forward advances the state through every chunk
        const int nsteps = (rev || helper || kFwd) ? c1 - c0 : c1 - c0 - 1;
        const bool prep = !(rev && split);  // this CTA builds Abar / M / T itself
        const bool need_m = rev || helper || kFwd;  // M is needed (reverse pass, or for it, or O)
        if (rev && !rebuild) {  // split mode: the last chunk's start state comes from scratch too
          if (tid == 0) {
            const uint8_t* slot = segbuf + static_cast<size_t>(c1 - 1 - c0) * sbytes;
            mbar_expect_tx(bar_a1, kStateBytes);
            bulk_load(sb + OFF_A1, slot, kStateBytes, bar_a1);
            load_prep(slot);
          }
          a1_pending = true;
          sm_pending = true;
        }
        // raw bf16 bits of beta: converted where used, so no thread waits on the load early
        unsigned short braw_next = 0;
        if (nsteps > 0) {  // first chunk of the pass: issue its loads now
          const int c = rev ? c1 - 1 : c0;
          const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
          const int rows = static_cast<int>(min(static_cast<int64_t>(kC), eos - t0));
          stage_tiles(a, sb + OFF_STG, h, t0, rows, tid, true, rev, sb + OFF_SDO, need_m);
          cp_async_commit();
          if (tid < kC && tid < rows) braw_next = beta_bits(a.b, (t0 + tid) * a.H + h);
        }
#pragma unroll 1
        for (int step = 0; step < nsteps; ++step) {
          const int c = rev ? c1 - 1 - step : c0 + step;
          const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
          const int rows = static_cast<int>(min(static_cast<int64_t>(kC), eos - t0));
          const int buf = step & 1;
          const uint8_t* SQ = sm + OFF_STG + buf * kStgBuf;
          const uint8_t* SK = SQ + 4096;
          const uint8_t* SV = SQ + 2 * 4096;
          const uint8_t* SG = SQ + 3 * 4096;
          const bool more = step + 1 < nsteps;
          const unsigned short braw = braw_next;
          // ---- prefetch the next chunk of this pass; save the start state ----
          if (more) {
            const int cn = rev ? c - 1 : c + 1;
            const int64_t tn = bos + static_cast<int64_t>(cn) * kC;
            const int rn = static_cast<int>(min(static_cast<int64_t>(kC), eos - tn));
            stage_tiles(a, sb + OFF_STG + (buf ^ 1) * kStgBuf, h, tn, rn, tid, true, false, 0, need_m);
            if (tid < kC && tid < rn) braw_next = beta_bits(a.b, (tn + tid) * a.H + h);
          }
          cp_async_commit();
          KDA_STAGE(BS_TILES_ISSUE);
          if constexpr (!kFwd) {
            if (!rev && tid == 0) bulk_store(segbuf + static_cast<size_t>(c - c0) * sbytes, sb + OFF_A1, kStateBytes);
          }
          KDA_STAGE(BS_STATE_STORE);
          cp_async_wait_prev();
          KDA_STAGE(BS_TILES_WAIT);
          __syncthreads();
          KDA_STAGE(BS_TOP_BARRIER);
          KDA_STAGE_STEP();

          // ================= chunk prologue =================
          if (tid < kC) S[S_BETA + tid] = tid < rows ? sigm(__bfloat162float(__ushort_as_bfloat16(braw))) : 0.f;
          {  // row norms: warp w -> rows 2w, 2w+1 (sums interleaved; lanes 0-3 finish them)
            float sk0 = 0.f, sk1 = 0.f, sq0 = 0.f, sq1 = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float y0 = stg(SK, 2 * warp, lane + 32 * e), y1 = stg(SK, 2 * warp + 1, lane + 32 * e);
              sk0 += y0 * y0;
              sk1 += y1 * y1;
              if (need_m) {  // the rebuild alone does not use q
                const float x0 = stg(SQ, 2 * warp, lane + 32 * e), x1 = stg(SQ, 2 * warp + 1, lane + 32 * e);
                sq0 += x0 * x0;
                sq1 += x1 * x1;
              }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              sk0 += __shfl_xor_sync(0xffffffffu, sk0, o);
              sk1 += __shfl_xor_sync(0xffffffffu, sk1, o);
              sq0 += __shfl_xor_sync(0xffffffffu, sq0, o);
              sq1 += __shfl_xor_sync(0xffffffffu, sq1, o);
            }
            if (lane < 4) {  // lane 0/1: k rows, lane 2/3: q rows
              const float v = lane == 0 ? sk0 : (lane == 1 ? sk1 : (lane == 2 ? sq0 : sq1));
              const float nrm = sqrtf(v + a.eps);
              const float inv = nrm > 0.f ? 1.f / nrm : 0.f;
              S[(lane < 2 ? S_IK0 : S_IQ0) + 2 * warp + (lane & 1)] = inv;
            }
          }
          {  // gate, per-half cumulative log2 decay
            float gv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) gv[j] = stg(SG, 8 * rh + j, ci);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float d = 8 * rh + j < rows ? Lg * sigm(expA * (gv[j] + dtb)) : 0.f;
              acc += d;
              gv[j] = acc;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) GS[(8 * rh + j) * kLd + ci] = gv[j];
            S[S_TOT + rh * 128 + ci] = acc;
          }
          __syncthreads();
          KDA_STAGE(BS_NORM_GATE);
          {  // full cumsum, gated operands
            const float carry = rh ? S[S_TOT + ci] : 0.f;
            const float gend = S[S_TOT + ci] + S[S_TOT + 128 + ci];
            const float gam = ex2(gend);
            if (rh == 0) {
              S[S_GEND + ci] = gend;
              S[S_GAM + ci] = gam;
            }
            float Gv[8], kv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              Gv[j] = GS[r * kLd + ci] + carry;
              kv[j] = stg(SK, r, ci) * S[S_IK0 + r];
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              const float G = Gv[j], kh = kv[j];
              const float e = ex2(G);
              GS[r * kLd + ci] = G;
              KG[r * kLd + ci] = kh * e;
              const float ki = kh * ex2(-G);
              KI[r * kLd + ci] = ki;
              st_h(sm + OFF_FKB, sw128_off(r, ci, 16), ki * gam);  // Kbar = kh e^{G_end - G}
              if (need_m) {
                const float qg = stg(SQ, r, ci) * S[S_IQ0 + r] * a.scale * e;
                QG[r * kLd + ci] = qg;
                if (rev) {
                  st_h(sm + OFF_FQG, sw128_off(r, ci, 16), qg);
                  // bf16 -> fp16 is exact for these magnitudes
                  st_h(sm + OFF_FDO, sw128_off(r, ci, 16), stg(SDO, r, ci));
                } else if constexpr (kFwd) {
                  st_h(sm + OFF_FQG, sw128_off(r, ci, 16), qg);
                }
              }
            }
          }
          // split mode: the tiles above feed the early dU~ product directly (the
          // Abar / M, inverse and W/U stages and their barriers are the helper's)
          if (!prep) fence_async_smem();
          __syncthreads();
          KDA_STAGE(BS_OPERANDS);
          if (!prep) {  // split mode: this chunk's Abar, T, T', M come from the helper
            if (!mbar_wait(bar_sm, ph_sm, a.status)) *s_fail = 1;
            ph_sm ^= 1u;
            sm_pending = false;
          }
          KDA_STAGE(BS_SLOT_WAIT);
          if (rev) {  // next chunk's dO (the dO staging tile has been consumed)
            if (more) stage_tiles(a, 0, h, t0 - kC, kC, tid, false, true, sb + OFF_SDO);
            cp_async_commit();
          }
          KDA_STAGE(BS_DO_ISSUE);
          // ================= Abar (and M) on tf32 tensor tiles =================
          // warp w: column block nt = w & 1, contraction half kh = (w >> 1) & 1, Abar (w < 4) or
          // M (w >= 4); the kh = 1 warps hand their partial sums over in S_DT1 / S_DT2 (free here)
          if (prep && warp < (need_m ? 8 : 4)) {
            const int nt = warp & 1, kh = (warp >> 1) & 1;
            const bool is_m = (warp >> 2) != 0;
            const float* X = is_m ? QG : KG;
            float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k0 = 64 * kh; k0 < 64 * kh + 64; k0 += 16) {  // two independent accumulator chains
              float fa[4], fb[2];
              ldA(fa, X, kLd, k0, fg, ft);
              ldBc(fb, KI, kLd, 8 * nt, k0, fg, ft);
              mma3(d, fa, fb);
              ldA(fa, X, kLd, k0 + 8, fg, ft);
              ldBc(fb, KI, kLd, 8 * nt, k0 + 8, fg, ft);
              mma3(d2, fa, fb);
            }
            float* part = S + (is_m ? S_DT2 : S_DT1);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              d[e] += d2[e];
              if (kh) part[(fg + 8 * (e >> 1)) * kSq + 8 * nt + 2 * ft + (e & 1)] = d[e];
            }
            named_bar_sync(1, need_m ? 256 : 128);
            if (kh == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] += part[(fg + 8 * (e >> 1)) * kSq + 8 * nt + 2 * ft + (e & 1)];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = fg + 8 * (e >> 1), s = 8 * nt + 2 * ft + (e & 1);
              if (!is_m) {
                S[S_AB + r * kSq + s] = s < r ? d[e] : 0.f;
              } else {
                const float mv = s <= r ? d[e] : 0.f;
                st_h(sm + OFF_FM, sw128_off(s, r, 16), mv);  // K-major B of dU~^T: row s, column r
                st_h(sm + OFF_FML, sw128_off(s, r, 16), lo_part(mv));
                if constexpr (kFwd) S[S_DM + r * kSq + s] = mv;  // fp32 M for the forward's M U~
              }
            }
            }
          }
          if (prep) {
            fence_async_smem();
            fence_before_sync();
            __syncthreads();
          }
          KDA_STAGE(BS_ABAR_M);
          // dU~^T = dO^T (Mhi + Mlo) + dH'^T Kbar^T needs no U~: issue it now (warp 4 is idle
          // during the inverse) so it runs under the inverse and the W/U stage
          if (rev && warp == 4 && lane == 0) {
            fence_after_sync();
            mma(tmem + TM_DU, desc_mn(D0, OFF_FDO, 2048, 0), desc_k(D0, OFF_FM, 16, 0, 0),
                idesc(128, 16, true, false), 0);
            mma(tmem + TM_DU, desc_mn(D0, OFF_FDO, 2048, 0), desc_k(D0, OFF_FML, 16, 0, 0),
                idesc(128, 16, true, false), 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma(tmem + TM_DU, desc_k(D0, OFF_A1D, 128, 0, ks), desc_k(D0, OFF_FKB, 16, 0, ks),
                  idesc(128, 16), 1);
            mma_commit(bar_du);
          }
          if (prep && warp == 0) {
            // T = (I + N)^-1 with N = diag(beta) Abar strictly lower, in 8 x 8 blocks: lane j < 16
            // solves column j of its diagonal block (T11 or T22) by forward substitution, then lane
            // j < 8 forms column j of T21 = -T22 N21 T11 (lanes 16-31 repeat lanes 0-15, unused)
            const int j = lane & 15, b8 = 8 * (j >> 3);
            float x[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = (b8 + k == j) ? 1.f : 0.f;
#pragma unroll
            for (int s2 = 0; s2 < 7; ++s2) {  // right-looking: x[s2] is final, eliminate it below
#pragma unroll
              for (int k = s2 + 1; k < 8; ++k)
                x[k] -= S[S_BETA + b8 + k] * S[S_AB + (b8 + k) * kSq + b8 + s2] * x[s2];
            }
            if (lane < 16) {
#pragma unroll
              for (int k = 0; k < 8; ++k) S[S_T + (b8 + k) * kSq + j] = x[k];
            }
            __syncwarp();
            float z[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) z[k] = 0.f;
            if (lane < 8) {
              float y[8];  // (N21 T11)[., j]
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                float acc = 0.f;
#pragma unroll
                for (int s3 = 0; s3 < 8; ++s3) acc += S[S_AB + (8 + k) * kSq + s3] * x[s3];
                y[k] = S[S_BETA + 8 + k] * acc;
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m <= k; ++m) acc += S[S_T + (8 + k) * kSq + 8 + m] * y[m];
                z[k] = -acc;
              }
            }
            if (lane < 16) {
              const float bj = S[S_BETA + j];
#pragma unroll
              for (int r = 0; r < 16; ++r) {
                const float t = ((r >> 3) == (j >> 3)) ? x[r & 7] : ((r >= 8) ? z[r - 8] : 0.f);
                S[S_T + r * kSq + j] = t;
                S[S_TP + r * kSq + j] = t * bj;
              }
            }
          }
          KDA_STAGE(BS_INVERSE);
          // -W and U~ are rewritten next: the previous step's copies of them (all
          // but this step's state copy) have been read out
          if (helper && tid == 0) bulk_wait_read_but<1>();
          if (prep) {
            fence_async_smem();
            __syncthreads();
          }
          if (helper) {  // hand this chunk's Abar, T, T' and M hi / lo to the reverse CTA
            if (tid == 0) {
              uint8_t* slot = segbuf + static_cast<size_t>(c - c0) * sbytes;
              bulk_store(slot + kStateBytes, sb + OFF_SMALL, kPrepSBytes);
              bulk_store(slot + kStateBytes + kPrepSBytes, sb + OFF_FM, kPrepMBytes);
            }
          }
          if (prep) {  // W = T' (Kh Gamma) -> -W fp16;  U = T' V -> fp32  (channels 16w .. 16w+15)
            float dw[2][4] = {}, du[2][4] = {};
#pragma unroll
            for (int k0 = 0; k0 < kC; k0 += 8) {
              float fa[4];
              ldA(fa, S + S_TP, kSq, k0, fg, ft);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                const int n0 = 16 * warp + 8 * nt;
                float fb[2], fv[2];
                ldBr(fb, KG, kLd, n0, k0, fg, ft);
                mma3(dw[nt], fa, fb);
                fv[0] = stg(SV, k0 + ft, n0 + fg);
                fv[1] = stg(SV, k0 + ft + 4, n0 + fg);
                mma2_bexact(du[nt], fa, fv);
              }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const int i = 16 * warp + 8 * nt + 2 * ft;
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                const int r = fg + 8 * hr;
                st_h2(sm + OFF_FW, sw128_off(r, i, 16), -dw[nt][2 * hr], -dw[nt][2 * hr + 1]);
                *reinterpret_cast<float2*>(UT + r * kLd + i) = make_float2(du[nt][2 * hr], du[nt][2 * hr + 1]);
              }
            }
          }
          if (prep) {
            fence_async_smem();
            fence_before_sync();
            KDA_SYNC_OR_BAIL();
          }
          KDA_STAGE(BS_WU);
          // ================= U~ = U - W H (tcgen05) =================
          if (a1_pending) {  // this chunk's start state, loaded during the prologue
            if (!mbar_wait(bar_a1, ph_a1, a.status)) *s_fail = 1;
            ph_a1 ^= 1u;
            a1_pending = false;
          }
          if (prep) {  // (split mode: the helper shipped -W and U~ with the chunk's matrices)
            if (tid == 0) {
              fence_after_sync();
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                mma(tmem + TM_D1, desc_k(D0, OFF_A1, 128, 0, ks), desc_k(D0, OFF_FW, 16, 0, ks),
                    idesc(128, 16), ks > 0);
              mma_commit(bar);
            }
            KDA_WAIT_MMA();
            KDA_STAGE(BS_UT_MMA);
          }
          if (rev) {
            if (!mbar_wait(bar_du, ph_du, a.status)) *s_fail = 1;
            ph_du ^= 1u;
            KDA_STAGE(BS_DUT_MMA);
          }
          fence_after_sync();
          {
            float x[8];
            if (prep) {
              tmem_ld8(tmem + tlane + TM_D1 + 8 * hh, x);  // lane = v, columns r
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r = 8 * hh + j;
                const float u = UT[r * kLd + L] + x[j];
                UT[r * kLd + L] = u;
                st_h(sm + OFF_FU, sw128_off(r, L, 16), u);
              }
            }
            if (rev) {
              tmem_ld8(tmem + tlane + TM_DU + 8 * hh, x);  // dU~^T: lane = v, columns r
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r = 8 * hh + j;
                DUT[r * kLd + L] = x[j];
                st_h(sm + OFF_FDU, sw128_off(r, L, 16), x[j]);
              }
            }
          }
          fence_async_smem();
          fence_before_sync();
          KDA_SYNC_OR_BAIL();

          KDA_STAGE(BS_READOUT);
          if (!rev) {
            if (helper) {  // hand -W and U~ over; the segment's last chunk advances no state
              if (tid == 0) ship_wu(segbuf + static_cast<size_t>(c - c0) * sbytes);
              if (c == c1 - 1) continue;
            }
            // ============ rebuild pass: H <- diag(gamma) H + Kbar^T U~ ============
            if (tid == 0) {
              fence_after_sync();
              mma(tmem + TM_D2, desc_mn(D0, OFF_FU, 2048, 0), desc_mn(D0, OFF_FKB, 2048, 0),
                  idesc(128, 128, true, true), 0);
              if constexpr (kFwd) {  // O^T's state part, H^T (Qh Gamma)^T (lane = v, columns r)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                  mma(tmem + TM_DQ, desc_k(D0, OFF_A1, 128, 0, ks), desc_k(D0, OFF_FQG, 16, 0, ks),
                      idesc(128, 16), ks > 0);
              } else if (helper) {
                // the scratch copy of A1 has been read out (a helper's three -W / U~
                // copies may still be in flight: the next step waits for those)
                bulk_wait_read_but<3>();
              } else {
                bulk_wait_read();
              }
              mma_commit(bar);
            }
            if constexpr (kFwd) {  // O's intra-chunk part M U~ (3xTF32, channels 16w .. 16w+15) into the dU~ tile
              float mu[2][4] = {};
#pragma unroll
              for (int k0 = 0; k0 < kC; k0 += 8) {
                float fa[4];
                ldA(fa, S + S_DM, kSq, k0, fg, ft);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                  float fb[2];
                  ldBr(fb, UT, kLd, 16 * warp + 8 * nt, k0, fg, ft);
                  mma3(mu[nt], fa, fb);
                }
              }
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                const int i = 16 * warp + 8 * nt + 2 * ft;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                  *reinterpret_cast<float2*>(DUT + (fg + 8 * hr) * kLd + i) = make_float2(mu[nt][2 * hr], mu[nt][2 * hr + 1]);
              }
            }
            KDA_WAIT_MMA();
            KDA_STAGE(BS_REBUILD_MMA);
            fence_after_sync();
            if constexpr (kFwd) {  // o = H^T (Qh Gamma)^T + (M U~)^T, rows 8 hh .. 8 hh + 7 of value channel L
              __syncthreads();
              float x[8];
              tmem_ld8(tmem + tlane + TM_DQ + 8 * hh, x);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int r = 8 * hh + j;
                if (r < rows) a.o[((t0 + r) * a.H + h) * kD + L] = __float2bfloat16_rn(x[j] + DUT[r * kLd + L]);
              }
            }
            // the forward's checkpoint: the chunk-start state every kCPS chunks
            float* ck = nullptr;
            if constexpr (kFwd) {
              if (a.ckpt_out != nullptr && c % kCPS == 0)
                ck = a.ckpt_out + (ckpt_slot(bos, n, c / kCPS) * a.H + h) * static_cast<int64_t>(kD * kD);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float hv[32], dv[32];
              tmem_ld32(tmem + tlane + TM_H + 64 * hh + 32 * half, hv);
              tmem_ld32(tmem + tlane + TM_D2 + 64 * hh + 32 * half, dv);
              if (ck != nullptr) {
#pragma unroll
                for (int j = 0; j < 32; ++j) ck[(64 * hh + 32 * half + j) * kD + L] = hv[j];
              }
              const float4* g4 = reinterpret_cast<const float4*>(S + S_GAM + 64 * hh + 32 * half);
#pragma unroll
              for (int j4 = 0; j4 < 8; ++j4) {
                const float4 gm = g4[j4];
                hv[4 * j4] = gm.x * hv[4 * j4] + dv[4 * j4];
                hv[4 * j4 + 1] = gm.y * hv[4 * j4 + 1] + dv[4 * j4 + 1];
                hv[4 * j4 + 2] = gm.z * hv[4 * j4 + 2] + dv[4 * j4 + 2];
                hv[4 * j4 + 3] = gm.w * hv[4 * j4 + 3] + dv[4 * j4 + 3];
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
            KDA_STAGE(BS_STATE_UPDATE);
            continue;
          }

          // ================= reverse pass: backward of chunk c =================
          // Three issuers (lane 0 of warps 0-2), one mbarrier each:
          // state increment (Qh Gamma)^T dO - W^T dU~, transposed: dO^T QG + dU~^T (-W),
          // and (H dO^T); (H dU~^T); (dH' U~^T) -- lanes = key index i
          if (lane == 0 && warp < 3) {
            fence_after_sync();
            if (warp == 0) {
              mma(tmem + TM_D2, desc_mn(D0, OFF_FDO, 2048, 0), desc_mn(D0, OFF_FQG, 2048, 0),
                  idesc(128, 128, true, true), 0);
              mma(tmem + TM_D2, desc_mn(D0, OFF_FDU, 2048, 0), desc_mn(D0, OFF_FW, 2048, 0),
                  idesc(128, 128, true, true), 1);
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                mma(tmem + TM_DQ, desc_mn(D0, OFF_A1, 16384, ks), desc_k(D0, OFF_FDO, 16, 0, ks),
                    idesc(128, 16, true, false), ks > 0);
              mma_commit(bar);
            } else if (warp == 1) {
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                mma(tmem + TM_DW, desc_mn(D0, OFF_A1, 16384, ks), desc_k(D0, OFF_FDU, 16, 0, ks),
                    idesc(128, 16, true, false), ks > 0);
              mma_commit(bar_g1);
            } else {
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)
                mma(tmem + TM_DK, desc_mn(D0, OFF_A1D, 16384, ks), desc_k(D0, OFF_FU, 16, 0, ks),
                    idesc(128, 16, true, false), ks > 0);
              mma_commit(bar_g2);
            }
          }
          // ---- work that needs only dU~ and U~ runs while the state MMAs do:
          // dM = dO U~^T (warps 0-3) and dU~ V^T (warps 4-7), warp w: column
          // block w & 1, contraction half (w >> 1) & 1; the second halves land
          // in the PR / DAB scratch matrices and are folded in [D1] ----
          {
            const int nt = warp & 1, kh = (warp >> 1) & 1;
            const bool is_dm = warp < 4;
            float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 64 * kh; kk < 64 * kh + 64; kk += 8) {
              float fa[4], fb[2];
              float(&acc)[4] = (kk & 8) ? d2 : d;  // two independent accumulator chains
              if (is_dm) {  // dO exact in tf32
                fa[0] = h16(sm + OFF_FDO, sw128_off(fg, kk + ft, 16));
                fa[1] = h16(sm + OFF_FDO, sw128_off(fg + 8, kk + ft, 16));
                fa[2] = h16(sm + OFF_FDO, sw128_off(fg, kk + ft + 4, 16));
                fa[3] = h16(sm + OFF_FDO, sw128_off(fg + 8, kk + ft + 4, 16));
                ldBc(fb, UT, kLd, 8 * nt, kk, fg, ft);
                mma2_aexact(acc, fa, fb);
              } else {  // V exact in tf32
                ldA(fa, DUT, kLd, kk, fg, ft);
                fb[0] = stg(SV, 8 * nt + fg, kk + ft);
                fb[1] = stg(SV, 8 * nt + fg, kk + ft + 4);
                mma2_bexact(acc, fa, fb);
              }
            }
            const int dst = is_dm ? (kh ? S_PR : S_DM) : (kh ? S_DAB : S_DT2);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = fg + 8 * (e >> 1), sc = 8 * nt + 2 * ft + (e & 1);
              S[dst + r * kSq + sc] = d[e] + d2[e];
            }
          }
          // the first and last chunk of a sequence also use the low part of
          // their start state (written by the rebuild pass with plain stores,
          // read past L1 in [E])
          const bool edge = kEdge && (c == 0 || c == nchunks - 1);
          KDA_STAGE(BS_DM);
          KDA_WAIT_MMA();
          KDA_STAGE(BS_STATE_MMA);
          if (!mbar_wait(bar_g1, ph_g1, a.status)) *s_fail = 1;
          ph_g1 ^= 1u;
          if (!mbar_wait(bar_g2, ph_g2, a.status)) *s_fail = 1;
          ph_g2 ^= 1u;
          fence_after_sync();
          if (edge)  // dgamma's low-part term for a sequence-edge chunk
            edge_dgamma_lo(edge_buf + (c == 0 ? 0 : kStateBytes), tmem + tlane + TM_DH + 64 * hh, L, hh, lane,
                           RED + 512 + q4 * 128 + 64 * hh);
          // ---- [E] dH update, dgamma (lane = v); dQG, dW, dKbar (lane = i) ----
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
              const float4* g4 = reinterpret_cast<const float4*>(S + S_GAM + 64 * hh + 32 * half);
#pragma unroll
              for (int j4 = 0; j4 < 8; ++j4) {
                const float4 gm = g4[j4];
                dh[4 * j4] = gm.x * dh[4 * j4] + inc[4 * j4];
                dh[4 * j4 + 1] = gm.y * dh[4 * j4 + 1] + inc[4 * j4 + 1];
                dh[4 * j4 + 2] = gm.z * dh[4 * j4 + 2] + inc[4 * j4 + 2];
                dh[4 * j4 + 3] = gm.w * dh[4 * j4 + 3] + inc[4 * j4 + 3];
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
              RED[q4 * 128 + 64 * hh + base] = p[0];
              RED[q4 * 128 + 64 * hh + base + 1] = p[1];
            }
            float xq[8], xw[8], xk[8];
            tmem_ld8(tmem + tlane + TM_DQ + 8 * hh, xq);  // lane = i, columns r
            tmem_ld8(tmem + tlane + TM_DW + 8 * hh, xw);
            tmem_ld8(tmem + tlane + TM_DK + 8 * hh, xk);
            const int i = L;
            const float gend = S[S_GEND + i], gam = S[S_GAM + i];
            float part = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * hh + j;
              const float G = GS[r * kLd + i];
              const float kbv = KI[r * kLd + i] * gam;
              AQ[r * kLd + i] = xq[j] * ex2(G);
              AG[r * kLd + i] = xq[j] * QG[r * kLd + i] - xk[j] * kbv;
              AK[r * kLd + i] = xk[j] * ex2(gend - G);
              WT[r * kLd + i] = -xw[j];  // dW
              part += xk[j] * kbv;
            }
            S[S_PART + hh * 128 + i] = part;
          }
          fence_async_smem();
          __syncthreads();
          if (edge) {  // add the low-part term of dgamma (RED2) to [E]'s partial sums
            edge_fold(RED);
            __syncthreads();
          }
          KDA_STAGE(BS_E);
          // the next chunk's start state into A1 (its last reader was [E])
          if (more) {
            if (tid == 0) {
              mbar_expect_tx(bar_a1, kStateBytes);
              bulk_load(sb + OFF_A1, segbuf + static_cast<size_t>(c - 1 - c0) * sbytes, kStateBytes, bar_a1);
            }
            a1_pending = true;
          }
          // ---- [D1] d(chunk-end log decay); dW (Kh Gamma)^T on tf32 tiles ----
          if (tid >= kD) {
            const int i = tid - kD;
            const float dgam = RED[i] + RED[128 + i] + RED[256 + i] + RED[384 + i];
            S[S_DGE + i] = S[S_PART + i] + S[S_PART + 128 + i] + dgam * S[S_GAM + i];
#pragma unroll
            for (int e = 0; e < 2; ++e) {  // fold the second contraction halves of dM and dU~ V^T
              const int x = 2 * i + e, r = x >> 4, sc = x & 15, o = r * kSq + sc;
              S[S_DM + o] = sc > r ? 0.f : S[S_DM + o] + S[S_PR + o];
              S[S_DT2 + o] += S[S_DAB + o];
            }
          } else {  // warps 0..3: column block nt, contraction half kh (partial sums in DT1 / Y)
            const int nt = warp & 1, kh = warp >> 1;
            float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 64 * kh; kk < 64 * kh + 64; kk += 16) {
              float fa[4], fb[2];
              ldA(fa, WT, kLd, kk, fg, ft);
              ldBc(fb, KG, kLd, 8 * nt, kk, fg, ft);
              mma3(d, fa, fb);
              ldA(fa, WT, kLd, kk + 8, fg, ft);
              ldBc(fb, KG, kLd, 8 * nt, kk + 8, fg, ft);
              mma3(d2, fa, fb);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = fg + 8 * (e >> 1), s = 8 * nt + 2 * ft + (e & 1);
              S[(kh ? S_Y : S_DT1) + r * kSq + s] = d[e] + d2[e];
            }
          }
          __syncthreads();
          KDA_STAGE(BS_D1);
          // ---- [D2] dT = dT' diag(beta) (strictly lower; dT' = DT1 + Y + DT2 partials),
          // Y = dT T^T and dA = -T^T Y on tf32 tiles, warp nt: columns 8nt .. 8nt+7 ----
          if (warp < 2) {
            const int nt = warp;
            float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k0 = 0; k0 < kC; k0 += 8) {
              float fa[4], fb[2];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int r = fg + 8 * (e & 1), b2 = k0 + ft + 4 * (e >> 1);
                const int x = r * kSq + b2;
                fa[e] = b2 < r ? (S[S_DT1 + x] + S[S_Y + x] + S[S_DT2 + x]) * S[S_BETA + b2] : 0.f;
              }
              ldBc(fb, S + S_T, kSq, 8 * nt, k0, fg, ft);  // B[b][s] = T[s][b]
              mma3(y, fa, fb);
            }
            float* Yw = S + S_DAB;  // this warp's columns of Y, then of diag(beta) dA
            Yw[fg * kSq + 8 * nt + 2 * ft] = y[0];
            Yw[fg * kSq + 8 * nt + 2 * ft + 1] = y[1];
            Yw[(fg + 8) * kSq + 8 * nt + 2 * ft] = y[2];
            Yw[(fg + 8) * kSq + 8 * nt + 2 * ft + 1] = y[3];
            __syncwarp();
            float da[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k0 = 0; k0 < kC; k0 += 8) {
              float fa[4], fb[2];
              ldAT(fa, S + S_T, kSq, k0, fg, ft);              // A[r][a] = T[a][r]
              ldBr(fb, Yw, kSq, 8 * nt, k0, fg, ft);           // B[a][s] = Y[a][s]
              mma3(da, fa, fb);
            }
            __syncwarp();
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = fg + 8 * (e >> 1), sc = 8 * nt + 2 * ft + (e & 1);
              const float d = sc < r ? -da[e] : 0.f;
              Yw[r * kSq + sc] = S[S_BETA + r] * d;
              S[S_PR + r * kSq + sc] = d * S[S_AB + r * kSq + sc];
            }
          } else if (warp == 2 && lane < kC) {  // dbeta from T' = T diag(beta)
            float db = 0.f;
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2) {
              const int x = r2 * kSq + lane;
              db += S[S_T + x] * (S[S_DT1 + x] + S[S_Y + x] + S[S_DT2 + x]);
            }
            S[S_DB + lane] = db;
          }
          __syncthreads();
          KDA_STAGE(BS_D2);
          if (tid < kC) {  // dbeta of rows: A = diag(beta) Abar
            float db = S[S_DB + tid];
#pragma unroll
            for (int s = 0; s < 16; ++s) db += S[S_PR + tid * kSq + s];
            S[S_DB + tid] = db;
          }
          {  // ---- [F] 16 x 128 gradient products (channels 16w .. 16w+15) ----
            float dvv[2][4] = {}, dkg[2][4] = {}, a1[2][4] = {}, m1[2][4] = {}, a2[2][4] = {};
#pragma unroll
            for (int k0 = 0; k0 < kC; k0 += 8) {
              float tpt[4], dab[4], dabt[4], dm[4], dmt[4];
              ldAT(tpt, S + S_TP, kSq, k0, fg, ft);
              ldA(dab, S + S_DAB, kSq, k0, fg, ft);
              ldAT(dabt, S + S_DAB, kSq, k0, fg, ft);
              ldA(dm, S + S_DM, kSq, k0, fg, ft);
              ldAT(dmt, S + S_DM, kSq, k0, fg, ft);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                const int n0 = 16 * warp + 8 * nt;
                float fb[2];
                ldBr(fb, DUT, kLd, n0, k0, fg, ft);
                mma1(dvv[nt], tpt, fb);  // dV = T'^T dU~ (feeds only dv: plain tf32)
                ldBr(fb, WT, kLd, n0, k0, fg, ft);
                mma3(dkg[nt], tpt, fb);  // d(Kh Gamma) += T'^T dW
                ldBr(fb, KI, kLd, n0, k0, fg, ft);
                mma3(a1[nt], dab, fb);  // (diag(beta) dA) (Kh / Gamma)
                mma3(m1[nt], dm, fb);   // dM (Kh / Gamma)
                ldBr(fb, KG, kLd, n0, k0, fg, ft);
                mma3(a2[nt], dabt, fb);  // (diag(beta) dA)^T (Kh Gamma)
                ldBr(fb, QG, kLd, n0, k0, fg, ft);
                mma3(a2[nt], dmt, fb);  // + dM^T (Qh Gamma)
              }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                const int r = fg + 8 * hr;
                const int i0 = 16 * warp + 8 * nt + 2 * ft;
                if (r < rows)
                  *reinterpret_cast<uint32_t*>(a.dv + ((t0 + r) * a.H + h) * kD + i0) =
                      pack_bf16(dvv[nt][2 * hr], dvv[nt][2 * hr + 1]);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int x = r * kLd + i0 + e, f = 2 * hr + e;
                  const float G = GS[x], eg = ex2(G), egi = ex2(-G);
                  const float kgp = dkg[nt][f] + a1[nt][f];
                  AQ[x] += m1[nt][f] * eg;
                  AK[x] += kgp * eg + a2[nt][f] * egi;
                  AG[x] += kgp * KG[x] + m1[nt][f] * QG[x] - a2[nt][f] * KI[x];
                }
              }
            }
          }
          fence_async_smem();
          __syncthreads();
          KDA_STAGE(BS_F);
          if (!prep && more) {  // the next chunk's Abar, T, T', M (last read in [D2] and [F])
            if (tid == 0) load_prep(segbuf + static_cast<size_t>(c - 1 - c0) * sbytes);
            sm_pending = true;
          }
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
          KDA_STAGE(BS_DG_CUMSUM);
          {  // L2-norm chain rule row dots: warp w -> rows 2w, 2w+1
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int r = 2 * warp + rr;
              float sq = 0.f, sk = 0.f;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = lane + 32 * e;
                sq += stg(SQ, r, i) * AQ[r * kLd + i];
                sk += stg(SK, r, i) * AK[r * kLd + i];
              }
              sq = warp_sum(sq);
              sk = warp_sum(sk);
              if (lane == 0) {
                S[S_RQ + r] = a.scale * sq * S[S_IQ0 + r];
                S[S_RK + r] = sk * S[S_IK0 + r];
              }
            }
          }
          __syncthreads();
          KDA_STAGE(BS_NORM_DOTS);
          {  // outputs dq, dk, dg (raw gate), parameter partials
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int r = 8 * rh + j;
              if (r < rows) {
                const int64_t off = ((t0 + r) * a.H + h) * kD + ci;
                const float iq0 = S[S_IQ0 + r], ik0 = S[S_IK0 + r];
                const float xq = stg(SQ, r, ci) * iq0, xk = stg(SK, r, ci) * ik0;
                a.dq[off] = __float2bfloat16_rn((a.scale * AQ[r * kLd + ci] - xq * S[S_RQ + r]) * iq0);
                a.dk[off] = __float2bfloat16_rn((AK[r * kLd + ci] - xk * S[S_RK + r]) * ik0);
                const float z = expA * (stg(SG, r, ci) + dtb);
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
          KDA_STAGE(BS_OUTPUTS);
        }
        if (kEdge && !rev) {
          // the rebuild pass leaves the start state of chunk c1 - 1 in TMEM:
          // when that is the sequence's last chunk, its low part goes to the
          // edge area (the first chunk's was stored with the checkpoint)
          if (c1 == nchunks && c1 - 1 > c0) {
            fence_after_sync();
            edge_lo_from_tmem(edge_buf + kStateBytes, tmem + tlane + TM_H + 64 * hh, L, hh);
          }
          __threadfence();  // the low parts went out as plain stores: visible before the publish
          __syncthreads();
        }
        if (!rev && tid == 0) {
          bulk_wait_all();  // scratch states written before pass 1 reads them
          if (helper) {
            fence_proxy_global();
            st_release(a.flags + kTcBwdFlags * item + lv % kTcBwdBufs, static_cast<uint32_t>(lv + 1));
          }
        }
        if (rev && split && tid == 0) st_release(a.flags + kTcBwdFlags * item + kTcBwdBufs, static_cast<uint32_t>(lv + 1));
        __syncthreads();
      }
    }

    if (helper) continue;
    if (seg > 0) {
      --seg;
      continue;
    }
    if constexpr (kFwd) {  // ---- forward item done: its final state ----
      if (a.hT != nullptr) {
        float* dst = a.hT + static_cast<int64_t>(item) * (kD * kD);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float x[32];
          tmem_ld32(tmem + tlane + TM_H + 64 * hh + 32 * half, x);
#pragma unroll
          for (int j = 0; j < 32; ++j) dst[(64 * hh + 32 * half + j) * kD + L] = x[j];
        }
      }
      __syncthreads();
      open = false;
      item += gridDim.x;
      continue;
    }
    // ---- item done: the gradient of the initial state (dH of the first chunk's start) ----
    if (a.dh0 != nullptr) {
      float* dst = a.dh0 + static_cast<int64_t>(item) * (kD * kD);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float x[32];
        tmem_ld32(tmem + tlane + TM_DH + 64 * hh + 32 * half, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(64 * hh + 32 * half + j) * kD + L] = x[j];
      }
    }
    // ---- and per-(sequence, head) partial sums of the gate-parameter gradients ----
    float* R = S + S_TOT;  // 256 floats
    R[tid] = acc_dtb;
    __syncthreads();
    if (tid < kD) a.partial[static_cast<int64_t>(item) * (kD + 1) + tid] = R[tid] + R[128 + tid];
    __syncthreads();
    R[tid] = acc_alog;
    __syncthreads();
    for (int st = kT / 2; st > 0; st >>= 1) {
      if (tid < st) R[tid] += R[tid + st];
      __syncthreads();
    }
    if (tid == 0) a.partial[static_cast<int64_t>(item) * (kD + 1) + kD] = R[0];
    __syncthreads();
    open = false;
    item += gridDim.x;
  }
#undef KDA_WAIT_MMA
#undef KDA_SYNC_OR_BAIL
teardown:
  // no async copy may still target this CTA's shared memory when it exits
  if (a1_pending) mbar_wait(bar_a1, ph_a1, a.status);
  if (sm_pending) mbar_wait(bar_sm, ph_sm, a.status);
  if (tid == 0) bulk_wait_all();
  asm volatile("cp.async.wait_all;" ::: "memory");
  fence_before_sync();
  __syncthreads();
  KDA_STAGE_FLUSH(g_bwd_stage);
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

size_t bwd_scratch_bytes_per_cta_tc() { return static_cast<size_t>(kCPS) * kSlotBytesInline; }
size_t bwd_scratch_bytes_per_buf_split_tc() { return static_cast<size_t>(kCPS) * kSlotBytesSplit; }
size_t bwd_edge_bytes_tc(int64_t items) { return static_cast<size_t>(items) * kEdgeBytes; }

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
  t.dhT = a.dhT;
  t.dh0 = a.dh0;
  t.dq = static_cast<__nv_bfloat16*>(a.dq);
  t.dk = static_cast<__nv_bfloat16*>(a.dk);
  t.dv = static_cast<__nv_bfloat16*>(a.dv);
  t.dg = static_cast<__nv_bfloat16*>(a.dg);
  t.db = static_cast<__nv_bfloat16*>(a.db);
  t.partial = a.partial;
  t.scratch = reinterpret_cast<uint8_t*>(a.scratch);
  t.edge = reinterpret_cast<uint8_t*>(a.edge);
  t.flags = a.flags;
  t.status = a.status;
  t.cu = a.cu;
  t.S = a.S;
  t.N = a.N;
  t.H = a.H;
  t.helpers = 0;
  t.scale = a.scale;
  t.lower = a.lower;
  t.eps = a.eps;
  t.o = nullptr;
  t.h0 = nullptr;
  t.hT = nullptr;
  t.ckpt_out = nullptr;
  const bool edge = a.dhT != nullptr || a.dh0 != nullptr;
  void (*kern)(const TcBwdArgs) = edge ? kda_bwd_tc_kernel<true, false> : kda_bwd_tc_kernel<false, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
    return KDA_ERR_CUDA;
  // Split mode: with fewer (sequence, head) items than SMs, the spare SMs
  // rebuild segment states for the reverse CTAs. Their hand-off waits need
  // every CTA resident at once, which a cooperative launch guarantees (or
  // refuses, and the inline mode runs instead).
  const int items = p->num_seqs * p->num_heads;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kT, SMEM_BYTES);
  int helpers = 0;
  if (a.flags != nullptr && items < kTcBwdCtas && items < sms) {
    const int spare = sms * per_sm - items;
    if (spare * 5 >= items * 2) helpers = spare < items ? spare : items;
  }
  bool launched = false;
  if (helpers > 0) {
    t.helpers = helpers;
    if (cudaMemsetAsync(a.flags, 0, sizeof(uint32_t) * (kTcBwdFlags * items + 1), s) != cudaSuccess)
      return KDA_ERR_CUDA;
    void* kargs[] = {&t};
    launched = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(items + helpers),
                                           dim3(kT), kargs, SMEM_BYTES, s) == cudaSuccess;
    if (!launched) {
      cudaGetLastError();  // clear the refusal; run inline instead
      t.helpers = 0;
    }
  }
  if (!launched && ctas > 0) kern<<<ctas, kT, SMEM_BYTES, s>>>(t);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  kda_param_reduce_tc_kernel<<<p->num_heads, 128, 0, s>>>(a.partial, p->num_seqs, p->num_heads, kD, a.dA_log,
                                                          a.ddt_bias);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// The forward with 16-token chunks: the backward kernel's forward mode, one CTA
// per SM walking its items' chunks in order (no helper CTAs, no scratch).
kda_status launch_fwd16_tc(const kda_problem* p, const FwdArgs& a, cudaStream_t s) {
  if (p->head_dim != kD || p->dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;
  TcBwdArgs t{};
  t.q = static_cast<const __nv_bfloat16*>(a.q);
  t.k = static_cast<const __nv_bfloat16*>(a.k);
  t.v = static_cast<const __nv_bfloat16*>(a.v);
  t.g = static_cast<const __nv_bfloat16*>(a.g);
  t.b = static_cast<const __nv_bfloat16*>(a.b);
  t.A_log = a.A_log;
  t.dt_bias = a.dt_bias;
  t.status = a.status;
  t.cu = a.cu;
  t.S = a.S;
  t.N = a.N;
  t.H = a.H;
  t.helpers = 0;
  t.scale = a.scale;
  t.lower = a.lower;
  t.eps = a.eps;
  t.o = static_cast<__nv_bfloat16*>(a.o);
  t.h0 = a.h0;
  t.hT = a.hT;
  t.ckpt_out = a.ckpt;
  void (*kern)(const TcBwdArgs) = kda_bwd_tc_kernel<false, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
    return KDA_ERR_CUDA;
  const int items = p->num_seqs * p->num_heads;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int ctas = items < sms ? items : sms;
  if (ctas > 0) kern<<<ctas, kT, SMEM_BYTES, s>>>(t);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
