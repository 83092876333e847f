// kda_simt.cu -- fp32 CUDA-core (SIMT) kernels for KDA forward and backward.
//
// These kernels evaluate the chunked KDA algorithm entirely in fp32 FFMA. They
// serve every dtype / head size the library accepts and are the path for fp32
// problems, whose tolerance (1e-4 relative) bf16 tensor-core operands cannot
// meet. The chunk decomposition follows "KDA at the production shape ...",
// section 2.1 (per-chunk ops: aqk, akk, w, u, v_new = u - w S, intra, inter,
// S += (k decay)^T v_new) and section 1.1 (serial state scan, channel-wise
// decay of the state). With chunk-local inclusive cumulative log-decay G_r
// (Gamma_r = exp(G_r), gamma = Gamma_{C-1}) and the chunk-start state H:
//   Abar[r,s] = sum_i kh_ri kh_si exp(G_ri - G_si)     (s < r)
//   M[r,s]    = sum_i qh_ri kh_si exp(G_ri - G_si)     (s <= r)
//   T = (I + diag(beta) Abar)^-1   (forward substitution)
//   W = T diag(beta) (Kh*Gamma),   U = T diag(beta) V
//   U~ = U - W H,   O = (Qh*Gamma) H + M U~,
//   H' = diag(gamma) H + Kbar^T U~,  Kbar[s,i] = kh_si exp(G_{C-1,i} - G_si).
// The factored products (kh*Gamma)(kh/Gamma)^T are safe in fp32 while the
// chunk's log-decay range stays below ~88 ("KDA at the production shape ...",
// section 3(a): the inverse-decay factor of k leaves fp32 range once the
// cumulative log-decay passes -88, which at the -5 floor limits a chunk to
// 17 tokens); these kernels use C = 16 (D = 64)
// and C = 8 (D = 128, to fit the backward's tiles in shared memory).
//
// GDN-2 (template flag CG, "KDA at the production shape ...", section 1.6
// and the section 2.1 op table): the scalar beta becomes a channel-wise erase
// gate Be[r,i] = sigmoid(erase_raw) on key channels and a write gate
// Wr[r,j] = sigmoid(write_raw) on value channels, so with Xw = Be*Kg and
// Xu = Wr*V the intra products read
//   Abar[r,s] = sum_i Xw_ri Ki_si (s < r),  T = (I + Abar)^-1,
//   W = T Xw,  U = T Xu,
// and everything after U~ = U - W H is unchanged (the state update writes
// kh r^T). KDA is the case Be = Wr = beta.
//
// Backward (recompute policy): the forward stores fp32 states every 1024
// tokens. For each such segment, in reverse order, the backward rebuilds the
// chunk-start states of the segment into per-CTA scratch with the same code
// the forward ran, then walks the segment's chunks in reverse: it recomputes
// the chunk's WY factors and gated q/k, propagates the state gradient dH,
// and writes dq, dk, dv, dg_raw, dbeta_raw once, in the input dtype.
#include <type_traits>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kNT = 256;

// Accumulator type of the contractions: fp64 for fp32 GDN-2 problems (see
// the backward kernel), fp32 otherwise.
template <typename Tin, bool CG>
struct AccOf {
  using type = float;
};
template <>
struct AccOf<float, true> {
  using type = double;
};

template <int D>
struct SimtChunk;
template <>
struct SimtChunk<64> {
  static constexpr int C = 16;
};
template <>
struct SimtChunk<128> {
  static constexpr int C = 8;
};

// Shared-memory tiles of one chunk. [C][LD] tiles use row stride LD = D + 1
// so that column walks by different threads hit different banks.
template <int D, int C>
struct Tiles {
  static constexpr int LD = D + 1, CP = C + 1, TILE = C * LD, SQ = C * CP;
  float *Qh, *Kh, *Gc, *Vv, *Qg, *Kg, *Ki, *Kb, *Ww, *Uu;
  float *Abar, *Aqk, *Tm;
  float *bet, *nq, *nk;
  float *gam, *dtb;
  float *Be, *Wr;  // GDN-2 only: erase gates [C][LD] (key channels), write gates [C][LD] (value channels)
  __device__ float* carve(float* p, bool cg = false) {
    Qh = p; p += TILE; Kh = p; p += TILE; Gc = p; p += TILE; Vv = p; p += TILE;
    Qg = p; p += TILE; Kg = p; p += TILE; Ki = p; p += TILE; Kb = p; p += TILE;
    Ww = p; p += TILE; Uu = p; p += TILE;
    Abar = p; p += SQ; Aqk = p; p += SQ; Tm = p; p += SQ;
    bet = p; p += C; nq = p; p += C; nk = p; p += C;
    gam = p; p += D; dtb = p; p += D;
    Be = Wr = nullptr;
    if (cg) {
      Be = p; p += TILE; Wr = p; p += TILE;
    }
    return p;
  }
  __host__ __device__ static constexpr int floats(bool cg = false) {
    return 10 * TILE + 3 * SQ + 3 * C + 2 * D + (cg ? 2 * TILE : 0);
  }
};

// dst[di(x)] = src[x] for x in [0, n): each thread issues kB of its global
// loads before any of its shared-memory stores, so their latencies overlap
// (in a plain copy loop every load waits behind the previous iteration's
// store, which the compiler cannot tell apart from the loaded address).
template <int kB, typename DstIdx>
__device__ __forceinline__ void load_batched(float* dst, const float* src, int n, DstIdx di) {
  for (int base = static_cast<int>(threadIdx.x); base < n; base += kNT * kB) {
    float tmp[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int x = base + j * kNT;
      tmp[j] = x < n ? src[x] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int x = base + j * kNT;
      if (x < n) dst[di(x)] = tmp[j];
    }
  }
}

// dst = src for n4 float4s (both 16-byte aligned), kB loads in flight per
// thread before its stores.
template <int kB>
__device__ __forceinline__ void copy4_batched(float* dst, const float* src, int n4) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
  float4* d4 = reinterpret_cast<float4*>(dst);
  for (int base = static_cast<int>(threadIdx.x); base < n4; base += kNT * kB) {
    float4 tmp[kB];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int x = base + j * kNT;
      if (x < n4) tmp[j] = s4[x];
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int x = base + j * kNT;
      if (x < n4) d4[x] = tmp[j];
    }
  }
}

// Loads rows [t0, t0 + rows) of head h (zeros beyond `rows`, which makes the
// padded rows inert: k = 0, beta = 0, g = 0) and builds
//   Qh = q/n_q (unscaled), Kh = k/n_k, Vv = v, bet = sigmoid(b),
//   Gc = chunk-local inclusive cumsum of g (natural-log units), gam = e^Gc[C-1],
//   Qg = scale*Qh*e^G, Kg = Kh*e^G, Ki = Kh*e^-G, Kb = Kh*e^(G[C-1]-G).
// G stays in natural-log units and every factor comes from expf: the
// exponential of a chunk-long sum amplifies the sum's absolute rounding into
// relative error, and a base-2 pre-scaling of each g by log2(e) would add
// one more rounding of that size (these kernels serve the fp32 problems,
// whose bar is 1e-4 of the RMS).
// The gate is g = lower * sigmoid(exp(A_log) * (g_raw + dt_bias)).
// With CG (GDN-2), b is the raw erase gate and w the raw write gate, both
// [S,H,D]: Be = sigmoid(b), Wr = sigmoid(w) (zero on padded rows) and bet is
// not used.
template <typename Tin, int D, int C, bool CG = false>
__device__ void chunk_prologue(const Tiles<D, C>& t, const Tin* q, const Tin* k, const Tin* v,
                               const Tin* g, const Tin* b, const Tin* w, int64_t t0, int rows, int h,
                               int H, float expA, float scale, float lower, float eps) {
  constexpr int LD = D + 1;
  constexpr int IT = C * D / kNT;  // elements per thread
  static_assert(C * D % kNT == 0, "the chunk tile must split evenly over the threads");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // all of this thread's global loads first, then the arithmetic and stores
  float qv[IT], kv[IT], vv[IT], gr[IT], br[CG ? IT : 1], wr[CG ? IT : 1];
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int x = tid + it * kNT, r = x / D, i = x % D;
    const int64_t off = ((t0 + r) * H + h) * (int64_t)D + i;
    const bool ok = r < rows;
    qv[it] = ok ? ldf(q + off) : 0.f;
    kv[it] = ok ? ldf(k + off) : 0.f;
    vv[it] = ok ? ldf(v + off) : 0.f;
    gr[it] = ok ? ldf(g + off) : 0.f;
    if constexpr (CG) {
      br[it] = ok ? ldf(b + off) : 0.f;
      wr[it] = ok ? ldf(w + off) : 0.f;
    }
  }
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int x = tid + it * kNT, r = x / D, i = x % D;
    const bool ok = r < rows;
    t.Qh[r * LD + i] = qv[it];
    t.Kh[r * LD + i] = kv[it];
    t.Gc[r * LD + i] = ok ? lower * sigmoidf_(expA * (gr[it] + t.dtb[i])) : 0.f;
    t.Vv[r * LD + i] = vv[it];
    if constexpr (CG) {
      t.Be[r * LD + i] = ok ? sigmoidf_(br[it]) : 0.f;
      t.Wr[r * LD + i] = ok ? sigmoidf_(wr[it]) : 0.f;
    }
  }
  if (!CG && tid < C) t.bet[tid] = tid < rows ? sigmoidf_(ldf(b + (t0 + tid) * H + h)) : 0.f;
  __syncthreads();
  for (int r = warp; r < C; r += kNT / 32) {
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < D; i += 32) {
      const float a = t.Qh[r * LD + i], c = t.Kh[r * LD + i];
      sq += a * a;
      sk += c * c;
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float nq = sqrtf(sq + eps), nk = sqrtf(sk + eps);
    // a zero row (padding, or eps = 0 with q = 0) stays exactly zero
    const float iq = nq > 0.f ? 1.f / nq : 0.f, ik = nk > 0.f ? 1.f / nk : 0.f;
    for (int i = lane; i < D; i += 32) {
      t.Qh[r * LD + i] *= iq;
      t.Kh[r * LD + i] *= ik;
    }
    if (lane == 0) {
      t.nq[r] = nq;
      t.nk[r] = nk;
    }
  }
  for (int i = tid; i < D; i += kNT) {
    float acc = 0.f;
    for (int r = 0; r < C; ++r) {
      acc += t.Gc[r * LD + i];
      t.Gc[r * LD + i] = acc;
    }
    t.gam[i] = expf(acc);
  }
  __syncthreads();
  for (int x = tid; x < C * D; x += kNT) {
    const int r = x / D, i = x % D;
    const float G = t.Gc[r * LD + i], Ge = t.Gc[(C - 1) * LD + i];
    const float e = expf(G), kh = t.Kh[r * LD + i];
    t.Qg[r * LD + i] = scale * t.Qh[r * LD + i] * e;
    t.Kg[r * LD + i] = kh * e;
    t.Ki[r * LD + i] = kh * expf(-G);
    t.Kb[r * LD + i] = kh * expf(Ge - G);
  }
  __syncthreads();
}

// Abar (strictly lower), Aqk (lower incl. diagonal), T = (I + diag(beta)Abar)^-1,
// W = T diag(beta) Kg, U = T diag(beta) V. With CG (GDN-2) Abar carries the
// erase gates, Abar[r,s] = sum_i Be_ri Kg_ri Ki_si, T = (I + Abar)^-1,
// W = T (Be*Kg) and U = T (Wr*V).
template <int D, int C, bool CG = false, typename Acc = float>
__device__ void chunk_intra(const Tiles<D, C>& t) {
  constexpr int LD = D + 1, CP = C + 1;
  constexpr int SP = kNT / (C * C);  // lanes per C x C output (contraction split over them)
  static_assert(SP >= 1 && C * C * SP == kNT && 32 % SP == 0, "one output per SP adjacent lanes");
  const int tid = threadIdx.x;
  {
    const int o = tid / SP, part = tid % SP, r = o / C, s = o % C;
    Acc akk = 0, aqk = 0;
    if (s <= r) {
      for (int i = part; i < D; i += SP) {
        const float ki = t.Ki[s * LD + i];
        if constexpr (CG)
          akk += Acc(t.Be[r * LD + i] * t.Kg[r * LD + i]) * ki;
        else
          akk += Acc(t.Kg[r * LD + i]) * ki;
        aqk += Acc(t.Qg[r * LD + i]) * ki;
      }
    }
#pragma unroll
    for (int m = 1; m < SP; m <<= 1) {
      akk += __shfl_xor_sync(0xffffffffu, akk, m);
      aqk += __shfl_xor_sync(0xffffffffu, aqk, m);
    }
    if (part == 0) {
      t.Abar[r * CP + s] = s < r ? static_cast<float>(akk) : 0.f;
      t.Aqk[r * CP + s] = s <= r ? static_cast<float>(aqk) : 0.f;
    }
  }
  __syncthreads();
  if (tid < 32) {  // forward substitution, one lane per column of T
    const int j = tid;
    for (int r = 0; r < C; ++r) {
      if (j < C) {
        Acc val;
        if (j == r) {
          val = 1;
        } else if (j > r) {
          val = 0;
        } else {
          val = 0;
          const float br = CG ? 1.f : t.bet[r];
          for (int s = j; s < r; ++s) val -= Acc(br * t.Abar[r * CP + s]) * t.Tm[s * CP + j];
        }
        t.Tm[r * CP + j] = static_cast<float>(val);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int x = tid; x < C * D; x += kNT) {
    const int r = x / D, i = x % D;
    Acc w = 0, u = 0;
    if constexpr (CG) {
      for (int s = 0; s <= r; ++s) {
        const Acc ts = t.Tm[r * CP + s];
        w += ts * (t.Be[s * LD + i] * t.Kg[s * LD + i]);
        u += ts * (t.Wr[s * LD + i] * t.Vv[s * LD + i]);
      }
    } else {
      for (int s = 0; s <= r; ++s) {
        const float ts = t.Tm[r * CP + s] * t.bet[s];
        w += ts * t.Kg[s * LD + i];
        u += ts * t.Vv[s * LD + i];
      }
    }
    t.Ww[r * LD + i] = static_cast<float>(w);
    t.Uu[r * LD + i] = static_cast<float>(u);
  }
  __syncthreads();
}

// U~ = U - W H (in place in Uu). H is D x V with row stride ldh.
template <int D, int C, typename Acc = float>
__device__ void state_residual(const Tiles<D, C>& t, const float* Hs, int ldh) {
  constexpr int V = D, LD = D + 1, RG = kNT / V, RPT = C / RG;
  static_assert(C % RG == 0, "rows per thread");
  const int tid = threadIdx.x, j = tid % V, rg = tid / V;
  Acc acc[RPT];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) acc[rr] = t.Uu[(rg * RPT + rr) * LD + j];
  for (int i = 0; i < D; ++i) {
    const float hv = Hs[i * ldh + j];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) acc[rr] -= Acc(t.Ww[(rg * RPT + rr) * LD + i]) * hv;
  }
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) t.Uu[(rg * RPT + rr) * LD + j] = static_cast<float>(acc[rr]);
  __syncthreads();
}

// H = diag(gam) H + Kb^T U~ (in place).
template <int D, int C, typename Acc = float>
__device__ void state_update(const Tiles<D, C>& t, float* Hs, int ldh) {
  constexpr int V = D, LD = D + 1, IG = kNT / V, IPT = D / IG;
  const int tid = threadIdx.x, j = tid % V, ig = tid / V;
  float u[C];
#pragma unroll
  for (int r = 0; r < C; ++r) u[r] = t.Uu[r * LD + j];
  for (int ii = 0; ii < IPT; ++ii) {
    const int i = ig * IPT + ii;
    Acc acc = Acc(t.gam[i]) * Hs[i * ldh + j];
#pragma unroll
    for (int r = 0; r < C; ++r) acc += Acc(t.Kb[r * LD + i]) * u[r];
    Hs[i * ldh + j] = static_cast<float>(acc);
  }
  __syncthreads();
}

// O = Qg H + Aqk U~, stored for rows < rows.
template <typename Tin, int D, int C>
__device__ void chunk_output(const Tiles<D, C>& t, const float* Hs, int ldh, Tin* o, int64_t t0,
                             int rows, int h, int H) {
  constexpr int V = D, LD = D + 1, CP = C + 1, RG = kNT / V, RPT = C / RG;
  const int tid = threadIdx.x, j = tid % V, rg = tid / V;
  float acc[RPT];
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) acc[rr] = 0.f;
  for (int i = 0; i < D; ++i) {
    const float hv = Hs[i * ldh + j];
#pragma unroll
    for (int rr = 0; rr < RPT; ++rr) acc[rr] += t.Qg[(rg * RPT + rr) * LD + i] * hv;
  }
#pragma unroll
  for (int rr = 0; rr < RPT; ++rr) {
    const int r = rg * RPT + rr;
    float a = acc[rr];
    for (int s = 0; s <= r; ++s) a += t.Aqk[r * CP + s] * t.Uu[s * LD + j];
    if (r < rows) stf(o + ((t0 + r) * H + h) * (int64_t)V + j, a);
  }
  __syncthreads();
}

template <typename Tin, int D, bool CG>
__global__ void __launch_bounds__(kNT, 1) kda_fwd_simt_kernel(const FwdArgs a) {
  constexpr int C = SimtChunk<D>::C, V = D;
  extern __shared__ float sm[];
  Tiles<D, C> t;
  float* Hs = t.carve(sm, CG);  // [D][V]
  const int n = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int64_t bos = a.cu[n], eos = a.cu[n + 1];
  const int tid = threadIdx.x;
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  const Tin* g = static_cast<const Tin*>(a.g);
  const Tin* b = static_cast<const Tin*>(a.b);
  const Tin* w = static_cast<const Tin*>(a.w);
  Tin* o = static_cast<Tin*>(a.o);
  for (int i = tid; i < D; i += kNT) t.dtb[i] = a.dt_bias[h * D + i];
  // initial state h0 [N][H][D][V] (zero when NULL)
  const float* h0 = a.h0 ? a.h0 + (int64_t)blockIdx.x * (D * V) : nullptr;
  if (h0 != nullptr)
    load_batched<8>(Hs, h0, D * V, [](int x) { return x; });
  else
    for (int x = tid; x < D * V; x += kNT) Hs[x] = 0.f;
  const float expA = expf(a.A_log[h]);
  __syncthreads();
  for (int64_t t0 = bos; t0 < eos; t0 += C) {
    const int64_t tt = t0 - bos;
    if (a.ckpt != nullptr && tt % kCkptTokens == 0) {
      float* dst = a.ckpt + (ckpt_slot(bos, n, (int)(tt / kCkptTokens)) * a.H + h) * (int64_t)(D * V);
      for (int x = tid; x < D * V; x += kNT) dst[x] = Hs[x];
    }
    const int rows = (int)min((int64_t)C, eos - t0);
    chunk_prologue<Tin, D, C, CG>(t, q, k, v, g, b, w, t0, rows, h, a.H, expA, a.scale, a.lower, a.eps);
    chunk_intra<D, C, CG>(t);
    state_residual<D, C>(t, Hs, V);
    chunk_output<Tin, D, C>(t, Hs, V, o, t0, rows, h, a.H);
    state_update<D, C>(t, Hs, V);
  }
  if (a.hT != nullptr) {  // final state
    __syncthreads();
    float* dst = a.hT + (int64_t)blockIdx.x * (D * V);
    for (int x = tid; x < D * V; x += kNT) dst[x] = Hs[x];
  }
}

// ---------------------------------------------------------------------------
// Backward
// ---------------------------------------------------------------------------
template <int D, int C>
struct BwdTiles {
  static constexpr int LD = D + 1, CP = C + 1, TILE = C * LD, SQ = C * CP, LDH = D + 1;
  float *dOt, *dUt, *dQ, *dK, *dGt, *dWt;  // [C][LD]
  float *dM, *dT, *Yt;                     // [C][CP]
  float *dbet, *rq, *rk;                   // [C]
  float *dGe, *part;                       // [D], [kNT]
  float *Hc, *dH;                          // [D][LDH]
  float *red;                              // [kNT]
  __device__ float* carve(float* p) {
    dOt = p; p += TILE; dUt = p; p += TILE; dQ = p; p += TILE; dK = p; p += TILE;
    dGt = p; p += TILE; dWt = p; p += TILE;
    dM = p; p += SQ; dT = p; p += SQ; Yt = p; p += SQ;
    dbet = p; p += C; rq = p; p += C; rk = p; p += C;
    dGe = p; p += D; part = p; p += kNT;
    Hc = p; p += D * LDH; dH = p; p += D * LDH;
    red = p; p += kNT;
    return p;
  }
  static constexpr int floats() { return 6 * TILE + 3 * SQ + 3 * C + D + 2 * kNT + 2 * D * LDH; }
  // Hc's offset in floats behind the chunk tiles: a multiple of 4, so that
  // Hc takes 16-byte copies (as does each D x LDH scratch slot)
  __host__ __device__ static constexpr int hc_offset(int tiles_floats) {
    return tiles_floats + 6 * TILE + 3 * SQ + 3 * C + D + kNT;
  }
};

template <typename Tin, int D, bool CG>
__global__ void __launch_bounds__(kNT, 1) kda_bwd_simt_kernel(const BwdArgs a) {
  constexpr int C = SimtChunk<D>::C, V = D, LD = D + 1, CP = C + 1, LDH = V + 1;
  constexpr int CPS = kCkptTokens / C;  // chunks per checkpoint segment
  constexpr int RGD = kNT / D, RPTD = C / RGD;
  extern __shared__ float sm[];
  // fp32 GDN-2 problems accumulate every contraction of the backward in fp64
  // (products of fp32 values are exact there; results are stored in fp32):
  // the erase-gate gradient takes two large terms through W and through
  // Abar that nearly cancel, and its 1e-4-of-RMS bar needs them to better
  // than fp32.
  using Acc = typename AccOf<Tin, CG>::type;
  static_assert(BwdTiles<D, C>::hc_offset(Tiles<D, C>::floats(CG)) % 4 == 0 && (D * LDH) % 4 == 0,
                "the state tile and its scratch slots must take 16-byte copies");
  Tiles<D, C> t;
  BwdTiles<D, C> u;
  u.carve(t.carve(sm, CG));
  const int tid = threadIdx.x;
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  const Tin* g = static_cast<const Tin*>(a.g);
  const Tin* b = static_cast<const Tin*>(a.b);
  const Tin* w = static_cast<const Tin*>(a.w);
  const Tin* dO = static_cast<const Tin*>(a.dO);
  Tin* dq = static_cast<Tin*>(a.dq);
  Tin* dk = static_cast<Tin*>(a.dk);
  Tin* dv = static_cast<Tin*>(a.dv);
  Tin* dg = static_cast<Tin*>(a.dg);
  Tin* db = static_cast<Tin*>(a.db);  // CG: gradient of the raw erase gate [S,H,D]
  Tin* dw = static_cast<Tin*>(a.dw);  // CG: gradient of the raw write gate [S,H,D]
  float* scratch = a.scratch + (int64_t)blockIdx.x * CPS * D * LDH;
  const int nitems = a.N * a.H;

  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int n = item / a.H, h = item % a.H;
    const int64_t bos = a.cu[n], eos = a.cu[n + 1];
    const int64_t T = eos - bos;
    const int nchunks = (int)((T + C - 1) / C);
    const int nseg = (int)((T + kCkptTokens - 1) / kCkptTokens);
    const float expA = expf(a.A_log[h]);
    for (int i = tid; i < D; i += kNT) t.dtb[i] = a.dt_bias[h * D + i];
    // dH = dhT, the gradient of the final state (zero when NULL)
    const float* dhT = a.dhT ? a.dhT + (int64_t)item * (D * V) : nullptr;
    if (dhT != nullptr) {
      for (int i = tid; i < D; i += kNT) u.dH[i * LDH + V] = 0.f;  // the padding column
      load_batched<8>(u.dH, dhT, D * V, [](int x) { return (x / V) * LDH + x % V; });
    } else {
      for (int x = tid; x < D * LDH; x += kNT) u.dH[x] = 0.f;
    }
    float acc_dtb = 0.f, acc_alog = 0.f;  // thread owns column tid % D
    __syncthreads();

    for (int seg = nseg - 1; seg >= 0; --seg) {
      const int c0 = seg * CPS, c1 = min(nchunks, c0 + CPS);
      {  // checkpoint -> Hc
        const float* src = a.ckpt + (ckpt_slot(bos, n, seg) * a.H + h) * (int64_t)(D * V);
        load_batched<8>(u.Hc, src, D * V, [](int x) { return (x / V) * LDH + x % V; });
      }
      __syncthreads();
      // rebuild the chunk-start states of this segment
      for (int c = c0; c < c1; ++c) {
        float* dst = scratch + (int64_t)(c - c0) * D * LDH;
        copy4_batched<4>(dst, u.Hc, D * LDH / 4);
        if (c == c1 - 1) break;
        const int64_t t0 = bos + (int64_t)c * C;
        const int rows = (int)min((int64_t)C, eos - t0);
        chunk_prologue<Tin, D, C, CG>(t, q, k, v, g, b, w, t0, rows, h, a.H, expA, a.scale, a.lower, a.eps);
        chunk_intra<D, C, CG, Acc>(t);
        state_residual<D, C, Acc>(t, u.Hc, LDH);
        state_update<D, C, Acc>(t, u.Hc, LDH);
      }
      __syncthreads();

      for (int c = c1 - 1; c >= c0; --c) {
        const int64_t t0 = bos + (int64_t)c * C;
        const int rows = (int)min((int64_t)C, eos - t0);
        {
          const float* src = scratch + (int64_t)(c - c0) * D * LDH;
          copy4_batched<9>(u.Hc, src, D * LDH / 4);
          constexpr int ITO = C * V / kNT;
          static_assert(C * V % kNT == 0, "the dO tile must split evenly over the threads");
          float dov[ITO];
#pragma unroll
          for (int it = 0; it < ITO; ++it) {
            const int x = tid + it * kNT, r = x / V, j = x % V;
            dov[it] = r < rows ? ldf(dO + ((t0 + r) * a.H + h) * (int64_t)V + j) : 0.f;
          }
#pragma unroll
          for (int it = 0; it < ITO; ++it) {
            const int x = tid + it * kNT, r = x / V, j = x % V;
            u.dOt[r * LD + j] = dov[it];
          }
        }
        chunk_prologue<Tin, D, C, CG>(t, q, k, v, g, b, w, t0, rows, h, a.H, expA, a.scale, a.lower, a.eps);
        chunk_intra<D, C, CG, Acc>(t);
        state_residual<D, C, Acc>(t, u.Hc, LDH);  // t.Uu = U~, t.Ww = W

        // dU~[r][j] = sum_{r'>=r} Aqk[r'][r] dO[r'][j] + sum_i Kb[r][i] dH[i][j]
        {
          constexpr int RG = kNT / V, RPT = C / RG;
          const int j = tid % V, rg = tid / V;
          Acc acc[RPT];
#pragma unroll
          for (int rr = 0; rr < RPT; ++rr) {
            const int r = rg * RPT + rr;
            Acc s_ = 0;
            for (int r2 = r; r2 < C; ++r2) s_ += Acc(t.Aqk[r2 * CP + r]) * u.dOt[r2 * LD + j];
            acc[rr] = s_;
          }
          for (int i = 0; i < D; ++i) {
            const float dh = u.dH[i * LDH + j];
#pragma unroll
            for (int rr = 0; rr < RPT; ++rr) acc[rr] += Acc(t.Kb[(rg * RPT + rr) * LD + i]) * dh;
          }
#pragma unroll
          for (int rr = 0; rr < RPT; ++rr) u.dUt[(rg * RPT + rr) * LD + j] = static_cast<float>(acc[rr]);
        }
        __syncthreads();

        // Terms that contract over the value dimension with H or dH:
        //   d(Qg) = dO H^T, dW = -dU~ H^T, dKb = U~ dH^T, dgamma = rowsum(H * dH)
        {
          const int i = tid % D, rg = tid / D;
          Acc aQ[RPTD], aW[RPTD], aK[RPTD], ag = 0;
#pragma unroll
          for (int rr = 0; rr < RPTD; ++rr) aQ[rr] = aW[rr] = aK[rr] = 0.f;
          for (int j = 0; j < V; ++j) {
            const float hv = u.Hc[i * LDH + j], dh = u.dH[i * LDH + j];
            ag += Acc(hv) * dh;
#pragma unroll
            for (int rr = 0; rr < RPTD; ++rr) {
              const int r = rg * RPTD + rr;
              aQ[rr] += Acc(u.dOt[r * LD + j]) * hv;
              aW[rr] += Acc(u.dUt[r * LD + j]) * hv;
              aK[rr] += Acc(t.Uu[r * LD + j]) * dh;
            }
          }
          Acc ge = 0;
#pragma unroll
          for (int rr = 0; rr < RPTD; ++rr) {
            const int r = rg * RPTD + rr;
            const float G = t.Gc[r * LD + i], Ge = t.Gc[(C - 1) * LD + i];
            u.dQ[r * LD + i] = static_cast<float>(aQ[rr] * expf(G));
            u.dGt[r * LD + i] = static_cast<float>(aQ[rr] * t.Qg[r * LD + i] - aK[rr] * t.Kb[r * LD + i]);
            u.dWt[r * LD + i] = static_cast<float>(-aW[rr]);
            u.dK[r * LD + i] = static_cast<float>(aK[rr] * expf(Ge - G));
            ge += aK[rr] * t.Kb[r * LD + i];
          }
          if (rg == 0) ge += ag * t.gam[i];
          u.part[tid] = static_cast<float>(ge);
        }
        __syncthreads();
        for (int i = tid; i < D; i += kNT) {
          float s_ = 0.f;
          for (int r = 0; r < RGD; ++r) s_ += u.part[r * D + i];
          u.dGe[i] = s_;
        }
        // dH <- diag(gam) dH + Qg^T dO - W^T dU~  (dH now refers to the chunk start)
        {
          constexpr int IG = kNT / V, IPT = D / IG;
          const int j = tid % V, ig = tid / V;
          float o_[C], du[C];
#pragma unroll
          for (int r = 0; r < C; ++r) {
            o_[r] = u.dOt[r * LD + j];
            du[r] = u.dUt[r * LD + j];
          }
          for (int ii = 0; ii < IPT; ++ii) {
            const int i = ig * IPT + ii;
            Acc acc = Acc(t.gam[i]) * u.dH[i * LDH + j];
#pragma unroll
            for (int r = 0; r < C; ++r) acc += Acc(t.Qg[r * LD + i]) * o_[r] - Acc(t.Ww[r * LD + i]) * du[r];
            u.dH[i * LDH + j] = static_cast<float>(acc);
          }
        }
        // dM = tril(dO U~^T);  dT = strictly-lower part of dW Xw^T + dU~ Xu^T
        // (each output's contractions split over SP adjacent lanes)
        {
          constexpr int SP = kNT / (C * C);
          static_assert(SP >= 1 && C * C * SP == kNT && 32 % SP == 0, "one output per SP adjacent lanes");
          const int o = tid / SP, part = tid % SP, r = o / C, s = o % C;
          Acc dm = 0, d1 = 0, d2 = 0;
          if (s <= r)
            for (int j = part; j < V; j += SP) dm += Acc(u.dOt[r * LD + j]) * t.Uu[s * LD + j];
          if (s < r) {
            if constexpr (CG) {  // dW Xw^T + dU~ Xu^T with the channel gates
              for (int i = part; i < D; i += SP)
                d1 += Acc(u.dWt[r * LD + i]) * (Acc(t.Be[s * LD + i]) * t.Kg[s * LD + i]);
              for (int j = part; j < V; j += SP)
                d2 += Acc(u.dUt[r * LD + j]) * (Acc(t.Wr[s * LD + j]) * t.Vv[s * LD + j]);
            } else {
              for (int i = part; i < D; i += SP) d1 += u.dWt[r * LD + i] * t.Kg[s * LD + i];
              for (int j = part; j < V; j += SP) d2 += u.dUt[r * LD + j] * t.Vv[s * LD + j];
            }
          }
#pragma unroll
          for (int m = 1; m < SP; m <<= 1) {
            dm += __shfl_xor_sync(0xffffffffu, dm, m);
            d1 += __shfl_xor_sync(0xffffffffu, d1, m);
            d2 += __shfl_xor_sync(0xffffffffu, d2, m);
          }
          if (part == 0) {
            Acc dt = 0;
            if (s < r) dt = CG ? d1 + d2 : Acc(t.bet[s]) * (d1 + d2);
            u.dM[r * CP + s] = static_cast<float>(dm);
            u.dT[r * CP + s] = static_cast<float>(dt);
          }
        }
        __syncthreads();
        // Y = dT T^T
        for (int x = tid; x < C * C; x += kNT) {
          const int a_ = x / C, s = x % C;
          Acc y = 0;
          const int bmax = min(s, a_ - 1);
          for (int bb = 0; bb <= bmax; ++bb) y += Acc(u.dT[a_ * CP + bb]) * t.Tm[s * CP + bb];
          u.Yt[a_ * CP + s] = static_cast<float>(y);
        }
        __syncthreads();
        // dA = -(T^T Y) on the strictly lower part (reuse dT for dA)
        for (int x = tid; x < C * C; x += kNT) {
          const int r = x / C, s = x % C;
          Acc da = 0;
          if (s < r)
            for (int a_ = r; a_ < C; ++a_) da -= Acc(t.Tm[a_ * CP + r]) * u.Yt[a_ * CP + s];
          u.dT[r * CP + s] = static_cast<float>(da);
        }
        // dXw = T^T dW (in place, by column); dXu = T^T dU~ (into dOt, free now)
        for (int x = tid; x < D + V; x += kNT) {
          float col[C];
          float* base = x < D ? (u.dWt + x) : (u.dUt + (x - D));
#pragma unroll
          for (int r = 0; r < C; ++r) col[r] = base[r * LD];
          float* out = x < D ? (u.dWt + x) : (u.dOt + (x - D));
#pragma unroll
          for (int r = 0; r < C; ++r) {
            Acc s_ = 0;
            for (int r2 = r; r2 < C; ++r2) s_ += Acc(t.Tm[r2 * CP + r]) * col[r2];
            out[r * LD] = static_cast<float>(s_);
          }
        }
        __syncthreads();
        // dv = beta dXu (CG: dv = Wr dXu and the raw write-gate gradient V dXu Wr (1 - Wr))
        for (int x = tid; x < C * V; x += kNT) {
          const int r = x / V, j = x % V;
          if (r < rows) {
            const int64_t off = ((t0 + r) * a.H + h) * (int64_t)V + j;
            if constexpr (CG) {
              const float wr = t.Wr[r * LD + j], dxu = u.dOt[r * LD + j];
              stf(dv + off, wr * dxu);
              stf(dw + off, t.Vv[r * LD + j] * dxu * sigmoid_grad(ldf(w + off)));
            } else {
              stf(dv + off, t.bet[r] * u.dOt[r * LD + j]);
            }
          }
        }
        // dbeta (before the beta-sigmoid): Xw, Xu and the beta factor of A
        if constexpr (!CG) {
          const int warp = tid >> 5, lane = tid & 31;
          for (int r = warp; r < C; r += kNT / 32) {
            float s_ = 0.f;
            for (int i = lane; i < D; i += 32)
              s_ += u.dWt[r * LD + i] * t.Kg[r * LD + i] + u.dOt[r * LD + i] * t.Vv[r * LD + i];
            for (int s = lane; s < r; s += 32) s_ += u.dT[r * CP + s] * t.Abar[r * CP + s];
            s_ = warp_sum(s_);
            if (lane == 0) u.dbet[r] = s_;
          }
        }
        // elementwise contributions of Xw, Abar and Aqk to dq^, dk^, dG
        for (int x = tid; x < C * D; x += kNT) {
          const int r = x / D, i = x % D;
          const float G = t.Gc[r * LD + i], e = expf(G), ei = expf(-G);
          const float dxw = u.dWt[r * LD + i];
          if constexpr (CG) {
            // dXw = T^T dW + dA Ki; Xw = Be*Kg gives dBe = Kg dXw and dKg = Be dXw;
            // dKi = dA^T Xw
            Acc a1 = 0, a2 = 0, m1 = 0, m2 = 0;
            for (int s = 0; s < r; ++s) a1 += Acc(u.dT[r * CP + s]) * t.Ki[s * LD + i];
            for (int s = r + 1; s < C; ++s) a2 += Acc(u.dT[s * CP + r]) * (Acc(t.Be[s * LD + i]) * t.Kg[s * LD + i]);
            for (int s = 0; s <= r; ++s) m1 += Acc(u.dM[r * CP + s]) * t.Ki[s * LD + i];
            for (int s = r; s < C; ++s) m2 += Acc(u.dM[s * CP + r]) * t.Qg[s * LD + i];
            const Acc be = t.Be[r * LD + i], kg = t.Kg[r * LD + i], dX = dxw + a1;
            u.dQ[r * LD + i] += static_cast<float>(m1 * e);
            u.dK[r * LD + i] += static_cast<float>(be * e * dX + (a2 + m2) * ei);
            u.dGt[r * LD + i] += static_cast<float>(be * dX * kg + m1 * t.Qg[r * LD + i] - (a2 + m2) * t.Ki[r * LD + i]);
            if (r < rows) {
              const int64_t off = ((t0 + r) * a.H + h) * (int64_t)D + i;
              stf(db + off, static_cast<float>(kg * dX * Acc(sigmoid_grad(ldf(b + off)))));
            }
            continue;
          }
          const float br = t.bet[r];
          float a1 = 0.f, a2 = 0.f, m1 = 0.f, m2 = 0.f;
          for (int s = 0; s < r; ++s) a1 += u.dT[r * CP + s] * t.Ki[s * LD + i];
          a1 *= br;
          for (int s = r + 1; s < C; ++s) a2 += t.bet[s] * u.dT[s * CP + r] * t.Kg[s * LD + i];
          for (int s = 0; s <= r; ++s) m1 += u.dM[r * CP + s] * t.Ki[s * LD + i];
          for (int s = r; s < C; ++s) m2 += u.dM[s * CP + r] * t.Qg[s * LD + i];
          u.dQ[r * LD + i] += m1 * e;
          u.dK[r * LD + i] += br * e * dxw + a1 * e + (a2 + m2) * ei;
          u.dGt[r * LD + i] += br * dxw * t.Kg[r * LD + i] + a1 * t.Kg[r * LD + i] +
                               m1 * t.Qg[r * LD + i] - (a2 + m2) * t.Ki[r * LD + i];
        }
        __syncthreads();
        // dG of the chunk end, then reverse cumulative sum -> dg (natural log units)
        for (int i = tid; i < D; i += kNT) {
          float acc = u.dGe[i];
          for (int r = C - 1; r >= 0; --r) {
            acc += u.dGt[r * LD + i];
            u.dGt[r * LD + i] = acc;
          }
        }
        // row dots for the L2-norm chain rule
        {
          const int warp = tid >> 5, lane = tid & 31;
          for (int r = warp; r < C; r += kNT / 32) {
            float sq = 0.f, sk = 0.f;
            for (int i = lane; i < D; i += 32) {
              sq += t.Qh[r * LD + i] * u.dQ[r * LD + i];
              sk += t.Kh[r * LD + i] * u.dK[r * LD + i];
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            if (lane == 0) {
              u.rq[r] = a.scale * sq;
              u.rk[r] = sk;
            }
          }
        }
        __syncthreads();
        for (int x = tid; x < C * D; x += kNT) {
          const int r = x / D, i = x % D;
          if (r < rows) {
            const int64_t off = ((t0 + r) * a.H + h) * (int64_t)D + i;
            const float dxq = a.scale * u.dQ[r * LD + i];
            const float iq = t.nq[r] > 0.f ? 1.f / t.nq[r] : 0.f;
            const float ik = t.nk[r] > 0.f ? 1.f / t.nk[r] : 0.f;
            stf(dq + off, (dxq - t.Qh[r * LD + i] * u.rq[r]) * iq);
            stf(dk + off, (u.dK[r * LD + i] - t.Kh[r * LD + i] * u.rk[r]) * ik);
            const float z = expA * (ldf(g + off) + t.dtb[i]);
            const float dz = u.dGt[r * LD + i] * a.lower * sigmoid_grad(z);
            stf(dg + off, expA * dz);
            acc_dtb += expA * dz;
            acc_alog += dz * z;
          }
        }
        if (!CG && tid < C && tid < rows) {
          stf(db + (t0 + tid) * a.H + h, u.dbet[tid] * sigmoid_grad(ldf(b + (t0 + tid) * a.H + h)));
        }
        __syncthreads();
      }
    }
    // per-(sequence, head) partial sums of the gate-parameter gradients
    u.red[tid] = acc_dtb;
    __syncthreads();
    for (int i = tid; i < D; i += kNT) {
      float s_ = 0.f;
      for (int r = 0; r < RGD; ++r) s_ += u.red[r * D + i];
      a.partial[(int64_t)item * (D + 1) + i] = s_;
    }
    __syncthreads();
    u.red[tid] = acc_alog;
    __syncthreads();
    for (int st = kNT / 2; st > 0; st >>= 1) {
      if (tid < st) u.red[tid] += u.red[tid + st];
      __syncthreads();
    }
    if (tid == 0) a.partial[(int64_t)item * (D + 1) + D] = u.red[0];
    if (a.dh0 != nullptr) {  // the gradient of the initial state
      float* dst = a.dh0 + (int64_t)item * (D * V);
      for (int x = tid; x < D * V; x += kNT) dst[x] = u.dH[(x / V) * LDH + (x % V)];
    }
    __syncthreads();
  }
}

// dA_log[h] = sum_n partial[n][h][D], ddt_bias[h][i] = sum_n partial[n][h][i],
// in a fixed order (deterministic).
__global__ void kda_param_reduce_kernel(const float* partial, int N, int H, int D, float* dA_log,
                                        float* ddt_bias) {
  const int h = blockIdx.x;
  for (int i = threadIdx.x; i <= D; i += blockDim.x) {
    float s = 0.f;
    for (int n = 0; n < N; ++n) s += partial[((int64_t)n * H + h) * (D + 1) + i];
    if (i < D)
      ddt_bias[h * D + i] = s;
    else
      dA_log[h] = s;
  }
}

template <typename Tin, int D, bool CG = false>
kda_status launch_fwd_t(const kda_problem* p, const FwdArgs& a, cudaStream_t s) {
  constexpr int C = SimtChunk<D>::C;
  const size_t smem = sizeof(float) * (Tiles<D, C>::floats(CG) + D * D);
  auto kern = kda_fwd_simt_kernel<Tin, D, CG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  const int grid = p->num_seqs * p->num_heads;
  if (grid > 0) kern<<<grid, kNT, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

template <int D>
int bwd_ctas(const kda_problem* p) {
  int items = p->num_seqs * p->num_heads;
  return items < kMaxBwdCtas ? items : kMaxBwdCtas;
}

template <typename Tin, int D, bool CG = false>
kda_status launch_bwd_t(const kda_problem* p, const BwdArgs& a, cudaStream_t s) {
  constexpr int C = SimtChunk<D>::C;
  const size_t smem = sizeof(float) * (Tiles<D, C>::floats(CG) + BwdTiles<D, C>::floats());
  auto kern = kda_bwd_simt_kernel<Tin, D, CG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int grid = bwd_ctas<D>(p);
  if (sms > 0 && grid > sms) grid = sms;  // one resident CTA per SM
  if (grid > 0) kern<<<grid, kNT, smem, s>>>(a);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  kda_param_reduce_kernel<<<p->num_heads, 128, 0, s>>>(a.partial, p->num_seqs, p->num_heads, D, a.dA_log,
                                                       a.ddt_bias);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

kda_status launch_fwd_simt(const kda_problem* p, const FwdArgs& a, cudaStream_t s) {
  const bool bf = p->dtype == KDA_DTYPE_BF16;
  if (p->flags & KDA_FLAG_CHANNEL_GATES) {
    if (p->head_dim == 64)
      return bf ? launch_fwd_t<__nv_bfloat16, 64, true>(p, a, s) : launch_fwd_t<float, 64, true>(p, a, s);
    if (p->head_dim == 128)
      return bf ? launch_fwd_t<__nv_bfloat16, 128, true>(p, a, s) : launch_fwd_t<float, 128, true>(p, a, s);
    return KDA_ERR_UNSUPPORTED;
  }
  if (p->head_dim == 64) return bf ? launch_fwd_t<__nv_bfloat16, 64>(p, a, s) : launch_fwd_t<float, 64>(p, a, s);
  if (p->head_dim == 128) return bf ? launch_fwd_t<__nv_bfloat16, 128>(p, a, s) : launch_fwd_t<float, 128>(p, a, s);
  return KDA_ERR_UNSUPPORTED;
}

kda_status launch_bwd_simt(const kda_problem* p, const BwdArgs& a, cudaStream_t s) {
  const bool bf = p->dtype == KDA_DTYPE_BF16;
  if (p->flags & KDA_FLAG_CHANNEL_GATES) {
    if (p->head_dim == 64)
      return bf ? launch_bwd_t<__nv_bfloat16, 64, true>(p, a, s) : launch_bwd_t<float, 64, true>(p, a, s);
    if (p->head_dim == 128)
      return bf ? launch_bwd_t<__nv_bfloat16, 128, true>(p, a, s) : launch_bwd_t<float, 128, true>(p, a, s);
    return KDA_ERR_UNSUPPORTED;
  }
  if (p->head_dim == 64) return bf ? launch_bwd_t<__nv_bfloat16, 64>(p, a, s) : launch_bwd_t<float, 64>(p, a, s);
  if (p->head_dim == 128) return bf ? launch_bwd_t<__nv_bfloat16, 128>(p, a, s) : launch_bwd_t<float, 128>(p, a, s);
  return KDA_ERR_UNSUPPORTED;
}

// Backward launch with a caller-chosen number of persistent CTAs (each CTA
// owns one per-CTA scratch slot). Used by the no-allocation entry point,
// whose fixed scratch buffer holds only a few slots.
kda_status launch_bwd_simt_ctas(const kda_problem* p, const BwdArgs& a, cudaStream_t s, int ctas) {
  const bool bf = p->dtype == KDA_DTYPE_BF16;
  if (ctas < 1) return KDA_ERR_WORKSPACE;
  auto run = [&](auto tin_tag, auto d_tag) -> kda_status {
    using Tin = decltype(tin_tag);
    constexpr int D = decltype(d_tag)::value;
    constexpr int C = SimtChunk<D>::C;
    const size_t smem = sizeof(float) * (Tiles<D, C>::floats() + BwdTiles<D, C>::floats());
    auto kern = kda_bwd_simt_kernel<Tin, D, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return KDA_ERR_CUDA;
    kern<<<ctas, kNT, smem, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    kda_param_reduce_kernel<<<p->num_heads, 128, 0, s>>>(a.partial, p->num_seqs, p->num_heads, D, a.dA_log,
                                                         a.ddt_bias);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  };
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (p->head_dim == 64) return bf ? run(__nv_bfloat16{}, D64{}) : run(float{}, D64{});
  if (p->head_dim == 128) return bf ? run(__nv_bfloat16{}, D128{}) : run(float{}, D128{});
  return KDA_ERR_UNSUPPORTED;
}

size_t bwd_scratch_bytes_per_cta_simt(const kda_problem* p) {
  const int D = p->head_dim;
  const int C = D == 64 ? SimtChunk<64>::C : SimtChunk<128>::C;
  return (size_t)(kCkptTokens / C) * D * (D + 1) * sizeof(float);
}

// Per-CTA scratch of the SIMT backward: the chunk-start states of one
// checkpoint segment, fp32 with padded rows.
size_t bwd_scratch_bytes_simt(const kda_problem* p, int* nctas) {
  const int D = p->head_dim;
  const int C = D == 64 ? SimtChunk<64>::C : SimtChunk<128>::C;
  int items = p->num_seqs * p->num_heads;
  const int ctas = items < kMaxBwdCtas ? items : kMaxBwdCtas;
  if (nctas) *nctas = ctas;
  return (size_t)ctas * (kCkptTokens / C) * D * (D + 1) * sizeof(float);
}

}  // namespace kda
