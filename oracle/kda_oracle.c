/*
 * kda_oracle.c -- plain fp64 CPU oracle for Kimi Delta Attention (KDA),
 * forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it. It shares no code with the CUDA library.
 *
 * What it computes (per sequence, per head; sequences are packed along the
 * token axis and delimited by cu_seqlens, heads are independent):
 *
 *   prologue ("KDA Memory with Recompute: FLA vs cuDNN Frontend FROST",
 *   section "Sources and measurement configuration": in-kernel Q/K L2
 *   normalisation, beta sigmoid, safe gate with lower bound -5 built from the
 *   raw gate, A_log and dt_bias):
 *     qh_t   = scale * q_t / sqrt(|q_t|^2 + eps)
 *     kh_t   =         k_t / sqrt(|k_t|^2 + eps)
 *     beta_t = sigmoid(b_t)
 *     z_t    = exp(A_log[h]) * (a_t + dt_bias[h,:])          (per channel)
 *     g_t    = L * sigmoid(z_t),  L = lower bound (-5)        (per channel)
 *     alpha_t = exp(g_t)
 *   The pages state only "safe gate with lower bound -5" from raw gate,
 *   A_log and dt_bias; the closed form above is this project's reading (the
 *   smooth bounded map). Parity of that mapping is unpinned by the pages.
 *
 *   recurrence (the KDA gated delta rule, state S is D x V; S_0 = h0, the
 *   initial state, zero unless given):
 *     S_t = (I - beta_t kh_t kh_t^T) Diag(alpha_t) S_{t-1} + beta_t kh_t v_t^T
 *     o_t = S_t^T qh_t
 *   written out with the obvious associativity so each step is O(D*V):
 *     P_t = Diag(alpha_t) S_{t-1};  r_t = v_t - P_t^T kh_t;
 *     S_t = P_t + beta_t kh_t r_t^T.
 *   ("KDA at the production shape ..." section 1.1 describes the same
 *   channel-wise decay of the state, "b_h1 *= exp2(b_gk_last1)", and the
 *   section 2.1 table lists the chunked form of exactly this recurrence.)
 *
 *   final state hT = S_T. backward: the exact reverse-time adjoint of the loop
 *   above, derived by hand. With Gb the adjoint of S_t (Gb = dhT, the
 *   gradient of the final state, after the last token; zero unless given):
 *     Gb    += qh_t dO_t^T ;   dqh_t = S_t dO_t
 *     dbeta_t = kh_t^T Gb r_t ;  dr = beta_t Gb^T kh_t ;  dv_t = dr
 *     dkh_t = beta_t Gb r_t - P_t dr
 *     dP    = Gb - kh_t dr^T ;  dalpha_t[i] = sum_j dP[i][j] S_{t-1}[i][j]
 *     Gb    = Diag(alpha_t) dP          (adjoint of S_{t-1})
 *   and after the first token dh0 = Gb, the gradient of the initial state;
 *   then the elementwise chain rule through the prologue. States S_{t-1}
 *   for the reverse loop are rebuilt segment by segment from states stored
 *   every SEG tokens (same recurrence, same order, so bit-identical).
 *
 * GDN-2 (gdn2_oracle_run): "KDA at the production shape ...", section 1.6,
 * names GDN-2 as this operator with the scalar beta replaced by a
 * channel-wise erase gate b_t and write gate w_t (KDA being the special
 * case), and its section 2.1 op table gives the chunked form:
 * akk = (b*k*Gamma)(k/Gamma)^T, w = M^-1 (b k*Gamma), u = M^-1 (w*v). The
 * token recurrence with that chunked form is
 *     S_t = (I - kh_t (b_t * kh_t)^T) Diag(alpha_t) S_{t-1} + kh_t (w_t * v_t)^T
 * with b_t = sigmoid(erase_raw_t) over key channels and w_t =
 * sigmoid(write_raw_t) over value channels (the sigmoid mirrors beta's; the
 * pages print no activation for the two gates). b_t = w_t = beta_t gives KDA.
 *
 * All arithmetic is IEEE double; inputs and outputs are double arrays (the
 * caller widens bf16/fp32 inputs, which is exact).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SEG 256 /* tokens between stored states in the reverse loop */

typedef struct {
  int num_seqs, H, D;
  const int64_t* cu;
  const double *q, *k, *v, *g, *b, *A_log, *dt_bias, *dO;
  /* GDN-2 (channel-wise gates): b is then the raw erase gate [S][H][D] and w
   * the raw write gate [S][H][V]; db / dw are their gradients */
  int channel_gates;
  const double* w;
  double* dw;
  const double *h0, *dhT; /* [num_seqs][H][D][V] or NULL (zero) */
  double *hT, *dh0;       /* [num_seqs][H][D][V] or NULL (not written) */
  double scale, lower, eps;
  double *o, *dq, *dk, *dv, *dg, *db;
  double* partial; /* [num_seqs][H][D+1]: ddt_bias[D], dA_log */
  int next_job;
  int njobs;
  int failed;
  pthread_mutex_t lock;
} job_t;

static double sigm(double x) {
  if (x >= 0) return 1.0 / (1.0 + exp(-x));
  double e = exp(x);
  return e / (1.0 + e);
}

/* Per-token prologue quantities for token index t (global), head h. */
typedef struct {
  double *qh, *kh, *xq, *xk, *z, *sg, *alpha, *vv;
  double *be, *wg; /* GDN-2 erase gate (key channels), write gate (value channels) */
  double nq, nk, beta;
} tok_t;

static void prologue(const job_t* J, int64_t t, int h, tok_t* P) {
  const int D = J->D, H = J->H;
  const int64_t base = (t * H + h) * (int64_t)D;
  double sq = 0, sk = 0;
  for (int i = 0; i < D; ++i) {
    double qi = J->q[base + i], ki = J->k[base + i];
    sq += qi * qi;
    sk += ki * ki;
  }
  P->nq = sqrt(sq + J->eps);
  P->nk = sqrt(sk + J->eps);
  const double eA = exp((double)J->A_log[h]);
  for (int i = 0; i < D; ++i) {
    P->xq[i] = J->q[base + i] / P->nq;
    P->xk[i] = J->k[base + i] / P->nk;
    P->qh[i] = J->scale * P->xq[i];
    P->kh[i] = P->xk[i];
    P->z[i] = eA * ((double)J->g[base + i] + (double)J->dt_bias[h * D + i]);
    P->sg[i] = sigm(P->z[i]);
    P->alpha[i] = exp(J->lower * P->sg[i]);
    P->vv[i] = J->v[base + i];
  }
  if (J->channel_gates) {
    for (int i = 0; i < D; ++i) {
      P->be[i] = sigm((double)J->b[base + i]);
      P->wg[i] = sigm((double)J->w[base + i]);
    }
    P->beta = 0;
  } else {
    P->beta = sigm((double)J->b[t * H + h]);
  }
}

/* One step of the recurrence in place: S <- P + beta kh r^T, with
 * P = Diag(alpha) S and r = v - P^T kh. r (length V) is returned. */
static void step(int D, double* S, const tok_t* P, double* r) {
  const int V = D;
  for (int i = 0; i < D; ++i) {
    double a = P->alpha[i];
    double* Si = S + (int64_t)i * V;
    for (int j = 0; j < V; ++j) Si[j] *= a;
  }
  for (int j = 0; j < V; ++j) r[j] = P->vv[j];
  for (int i = 0; i < D; ++i) {
    double ki = P->kh[i];
    const double* Si = S + (int64_t)i * V;
    for (int j = 0; j < V; ++j) r[j] -= Si[j] * ki;
  }
  for (int i = 0; i < D; ++i) {
    double c = P->beta * P->kh[i];
    double* Si = S + (int64_t)i * V;
    for (int j = 0; j < V; ++j) Si[j] += c * r[j];
  }
}

/* GDN-2 step in place ("KDA at the production shape ...", section 1.6: the
 * scalar beta becomes a channel-wise erase gate b_t and write gate w_t; the
 * section 2.1 op table puts b on the key side of akk and w on v in u):
 *   P = Diag(alpha) S;  r = w * v - P^T (b * kh);  S <- P + kh r^T,
 * i.e. S_t = (I - kh (b * kh)^T) Diag(alpha) S_{t-1} + kh (w * v)^T. */
static void step_cg(int D, double* S, const tok_t* P, double* r) {
  const int V = D;
  for (int i = 0; i < D; ++i) {
    double a = P->alpha[i];
    double* Si = S + (int64_t)i * V;
    for (int j = 0; j < V; ++j) Si[j] *= a;
  }
  for (int j = 0; j < V; ++j) r[j] = P->wg[j] * P->vv[j];
  for (int i = 0; i < D; ++i) {
    double ke = P->be[i] * P->kh[i];
    const double* Si = S + (int64_t)i * V;
    for (int j = 0; j < V; ++j) r[j] -= Si[j] * ke;
  }
  for (int i = 0; i < D; ++i) {
    double ki = P->kh[i];
    double* Si = S + (int64_t)i * V;
    for (int j = 0; j < V; ++j) Si[j] += ki * r[j];
  }
}

static int run_one(job_t* J, int n, int h) {
  const int D = J->D, V = J->D, H = J->H;
  const int64_t bos = J->cu[n], eos = J->cu[n + 1];
  const int64_t T = eos - bos;
  const int64_t DV = (int64_t)D * V;
  const int64_t soff = ((int64_t)n * H + h) * DV; /* this (sequence, head)'s state */
  if (T <= 0) { /* no tokens: hT = h0 and dh0 = dhT */
    for (int64_t x = 0; x < DV; ++x) {
      if (J->hT) J->hT[soff + x] = J->h0 ? J->h0[soff + x] : 0.0;
      if (J->dh0) J->dh0[soff + x] = J->dhT ? J->dhT[soff + x] : 0.0;
    }
    return 0;
  }
  const int64_t nseg = (T + SEG - 1) / SEG;
  const int want_bwd = J->dO != NULL;

  double* S = calloc(DV, sizeof(double));
  double* ckpt = want_bwd ? malloc(sizeof(double) * DV * nseg) : NULL;
  double* segS = want_bwd ? malloc(sizeof(double) * DV * SEG) : NULL;
  double* Gb = want_bwd ? calloc(DV, sizeof(double)) : NULL;
  double* dP = want_bwd ? malloc(sizeof(double) * DV) : NULL;
  double* work = malloc(sizeof(double) * (20 * (int64_t)D + 64));
  if (!S || !work || (want_bwd && (!ckpt || !segS || !Gb || !dP))) {
    free(S); free(ckpt); free(segS); free(Gb); free(dP); free(work);
    return -1;
  }
  tok_t P;
  P.qh = work; P.kh = work + D; P.xq = work + 2 * D; P.xk = work + 3 * D;
  P.z = work + 4 * D; P.sg = work + 5 * D; P.alpha = work + 6 * D;
  P.vv = work + 7 * D;
  double* r = work + 8 * D;
  double* dO = work + 9 * D;
  double* dr = work + 10 * D;
  double* Gr = work + 11 * D;
  double* dqh = work + 12 * D;
  double* dkh = work + 13 * D;
  double* dalpha = work + 14 * D;
  P.be = work + 15 * D;
  P.wg = work + 16 * D;
  double* dke = work + 17 * D;
  void (*advance)(int, double*, const tok_t*, double*) = J->channel_gates ? step_cg : step;

  if (J->h0) memcpy(S, J->h0 + soff, sizeof(double) * DV);
  if (want_bwd && J->dhT) memcpy(Gb, J->dhT + soff, sizeof(double) * DV);

  /* ---------------- forward ---------------- */
  for (int64_t tt = 0; tt < T; ++tt) {
    if (want_bwd && tt % SEG == 0) memcpy(ckpt + (tt / SEG) * DV, S, sizeof(double) * DV);
    const int64_t t = bos + tt;
    prologue(J, t, h, &P);
    advance(D, S, &P, r);
    if (J->o) {
      double* o = J->o + (t * H + h) * (int64_t)V;
      for (int j = 0; j < V; ++j) o[j] = 0;
      for (int i = 0; i < D; ++i) {
        const double qi = P.qh[i];
        const double* Si = S + (int64_t)i * V;
        for (int j = 0; j < V; ++j) o[j] += Si[j] * qi;
      }
    }
  }

  if (J->hT) memcpy(J->hT + soff, S, sizeof(double) * DV);

  /* ---------------- backward ---------------- */
  if (want_bwd) {
    double dAlog = 0;
    double* ddtb = J->partial + ((int64_t)n * H + h) * (D + 1);
    for (int i = 0; i < D; ++i) ddtb[i] = 0;
    const double eA = exp((double)J->A_log[h]);
    for (int64_t seg = nseg - 1; seg >= 0; --seg) {
      const int64_t t0 = seg * SEG;
      const int64_t t1 = (t0 + SEG < T) ? t0 + SEG : T;
      /* rebuild S_{t-1} for t in [t0, t1) */
      memcpy(segS, ckpt + seg * DV, sizeof(double) * DV);
      for (int64_t tt = t0; tt + 1 < t1; ++tt) {
        double* nxt = segS + (tt - t0 + 1) * DV;
        memcpy(nxt, segS + (tt - t0) * DV, sizeof(double) * DV);
        prologue(J, bos + tt, h, &P);
        advance(D, nxt, &P, r);
      }
      for (int64_t tt = t1 - 1; tt >= t0; --tt) {
        const int64_t t = bos + tt;
        const double* Sp = segS + (tt - t0) * DV; /* S_{t-1} */
        prologue(J, t, h, &P);
        /* S_t (into dP as scratch) and r */
        memcpy(dP, Sp, sizeof(double) * DV);
        advance(D, dP, &P, r);
        const double* dOt = J->dO + (t * H + h) * (int64_t)V;
        for (int j = 0; j < V; ++j) dO[j] = dOt[j];
        /* dqh = S_t dO */
        for (int i = 0; i < D; ++i) {
          const double* Si = dP + (int64_t)i * V;
          double acc = 0;
          for (int j = 0; j < V; ++j) acc += Si[j] * dO[j];
          dqh[i] = acc;
        }
        /* Gb += qh dO^T */
        for (int i = 0; i < D; ++i) {
          double* Gi = Gb + (int64_t)i * V;
          const double qi = P.qh[i];
          for (int j = 0; j < V; ++j) Gi[j] += qi * dO[j];
        }
        if (J->channel_gates) {
          /* GDN-2 adjoint of step_cg (derived by hand):
           *   dkh = Gb r + b * dke,  dr = Gb^T kh,  dv = w * dr,  dw = v * dr,
           *   dke = -P dr,  db = kh * dke,  dP = Gb - (b * kh) dr^T,
           *   dalpha[i] = sum_j dP[i][j] S_{t-1}[i][j],  Gb <- Diag(alpha) dP */
          for (int j = 0; j < V; ++j) dr[j] = 0;
          for (int i = 0; i < D; ++i) {
            const double* Gi = Gb + (int64_t)i * V;
            double acc = 0;
            for (int j = 0; j < V; ++j) acc += Gi[j] * r[j];
            Gr[i] = acc;
            const double ki = P.kh[i];
            for (int j = 0; j < V; ++j) dr[j] += Gi[j] * ki;
          }
          for (int i = 0; i < D; ++i) {
            const double* Si = Sp + (int64_t)i * V;
            double acc = 0;
            for (int j = 0; j < V; ++j) acc += Si[j] * dr[j];
            dke[i] = -P.alpha[i] * acc;
            dkh[i] = Gr[i] + P.be[i] * dke[i];
          }
          for (int i = 0; i < D; ++i) {
            double* Gi = Gb + (int64_t)i * V;
            const double* Si = Sp + (int64_t)i * V;
            const double ke = P.be[i] * P.kh[i];
            double acc = 0;
            for (int j = 0; j < V; ++j) {
              const double d = Gi[j] - ke * dr[j];
              acc += d * Si[j];
              Gi[j] = P.alpha[i] * d;
            }
            dalpha[i] = acc;
          }
          const int64_t base = (t * H + h) * (int64_t)D;
          for (int i = 0; i < D; ++i) {
            const double dbe = P.kh[i] * dke[i];
            J->db[base + i] = dbe * P.be[i] * (1.0 - P.be[i]);
            const double dwg = P.vv[i] * dr[i];
            J->dw[base + i] = dwg * P.wg[i] * (1.0 - P.wg[i]);
            dr[i] *= P.wg[i]; /* dv */
          }
        } else {
          /* Gr = Gb r ; dbeta = kh^T Gr ; dr = beta Gb^T kh */
          double dbeta = 0;
          for (int j = 0; j < V; ++j) dr[j] = 0;
          for (int i = 0; i < D; ++i) {
            const double* Gi = Gb + (int64_t)i * V;
            double acc = 0;
            for (int j = 0; j < V; ++j) acc += Gi[j] * r[j];
            Gr[i] = acc;
            dbeta += P.kh[i] * acc;
            const double ki = P.kh[i];
            for (int j = 0; j < V; ++j) dr[j] += Gi[j] * ki;
          }
          for (int j = 0; j < V; ++j) dr[j] *= P.beta;
          /* dkh = beta Gr - P dr, with P = Diag(alpha) S_{t-1} */
          for (int i = 0; i < D; ++i) {
            const double* Si = Sp + (int64_t)i * V;
            double acc = 0;
            for (int j = 0; j < V; ++j) acc += Si[j] * dr[j];
            dkh[i] = P.beta * Gr[i] - P.alpha[i] * acc;
          }
          /* dP = Gb - kh dr^T ; dalpha = rowsum(dP .* S_{t-1}) ; Gb = Diag(alpha) dP */
          for (int i = 0; i < D; ++i) {
            double* Gi = Gb + (int64_t)i * V;
            const double* Si = Sp + (int64_t)i * V;
            const double ki = P.kh[i];
            double acc = 0;
            for (int j = 0; j < V; ++j) {
              const double d = Gi[j] - ki * dr[j];
              acc += d * Si[j];
              Gi[j] = P.alpha[i] * d;
            }
            dalpha[i] = acc;
          }
          J->db[t * H + h] = dbeta * P.beta * (1.0 - P.beta);
        }
        /* elementwise chain rule through the prologue */
        const int64_t base = (t * H + h) * (int64_t)D;
        double xdq = 0, xdk = 0;
        for (int i = 0; i < D; ++i) {
          xdq += P.xq[i] * (J->scale * dqh[i]);
          xdk += P.xk[i] * dkh[i];
        }
        for (int i = 0; i < D; ++i) {
          const double dxq = J->scale * dqh[i];
          J->dq[base + i] = (dxq - P.xq[i] * xdq) / P.nq;
          J->dk[base + i] = (dkh[i] - P.xk[i] * xdk) / P.nk;
          J->dv[base + i] = dr[i];
          const double dgi = dalpha[i] * P.alpha[i];          /* d/dg of exp(g)   */
          const double dz = dgi * J->lower * P.sg[i] * (1.0 - P.sg[i]);
          J->dg[base + i] = eA * dz;                           /* d/da             */
          ddtb[i] += eA * dz;                                  /* d/d dt_bias      */
          dAlog += dz * P.z[i];                                /* d/d A_log        */
        }
      }
    }
    ddtb[D] = dAlog;
    if (J->dh0) memcpy(J->dh0 + soff, Gb, sizeof(double) * DV);
  }
  free(S); free(ckpt); free(segS); free(Gb); free(dP); free(work);
  return 0;
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int job = J->next_job++;
    pthread_mutex_unlock(&J->lock);
    if (job >= J->njobs) break;
    if (run_one(J, job / J->H, job % J->H) != 0) {
      pthread_mutex_lock(&J->lock);
      J->failed = 1;
      pthread_mutex_unlock(&J->lock);
    }
  }
  return NULL;
}

static int oracle_run(int num_seqs, const int64_t* cu_seqlens, int H, int D, const double* q,
                      const double* k, const double* v, const double* g, const double* b,
                      const double* w, const double* A_log, const double* dt_bias, double scale,
                      double lower_bound, double eps, const double* dO, double* o, double* dq,
                      double* dk, double* dv, double* dg, double* db, double* dw, double* dA_log,
                      double* ddt_bias, const double* h0, double* hT, const double* dhT,
                      double* dh0, int num_threads, int channel_gates) {
  if (num_seqs < 0 || H <= 0 || D <= 0 || !cu_seqlens) return -1;
  for (int n = 0; n < num_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  if (dO && (!dq || !dk || !dv || !dg || !db || !dA_log || !ddt_bias)) return -1;
  if (channel_gates && (!w || (dO && !dw))) return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.num_seqs = num_seqs; J.H = H; J.D = D; J.cu = cu_seqlens;
  J.q = q; J.k = k; J.v = v; J.g = g; J.b = b; J.A_log = A_log; J.dt_bias = dt_bias;
  J.channel_gates = channel_gates; J.w = w; J.dw = dw;
  J.dO = dO; J.scale = scale; J.lower = lower_bound; J.eps = eps;
  J.o = o; J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.db = db;
  J.h0 = h0; J.hT = hT; J.dhT = dO ? dhT : NULL; J.dh0 = dO ? dh0 : NULL;
  J.njobs = num_seqs * H;
  if (dO) {
    J.partial = calloc((size_t)num_seqs * H * (D + 1) + 1, sizeof(double));
    if (!J.partial) return -2;
  }
  pthread_mutex_init(&J.lock, NULL);
  if (num_threads < 1) num_threads = 1;
  if (num_threads > J.njobs) num_threads = J.njobs > 0 ? J.njobs : 1;
  pthread_t* th = malloc(sizeof(pthread_t) * num_threads);
  int started = 0;
  for (int i = 1; th && i < num_threads; ++i)
    if (pthread_create(&th[started], NULL, worker, &J) == 0) ++started;
  worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&J.lock);
  if (dO) {
    /* fixed-order sum over sequences of the per-(sequence, head) partials */
    for (int h = 0; h < H; ++h) {
      double sa = 0;
      for (int i = 0; i < D; ++i) ddt_bias[h * D + i] = 0;
      for (int n = 0; n < num_seqs; ++n) {
        const double* p = J.partial + ((int64_t)n * H + h) * (D + 1);
        for (int i = 0; i < D; ++i) ddt_bias[h * D + i] += p[i];
        sa += p[D];
      }
      dA_log[h] = sa;
    }
    free(J.partial);
  }
  return J.failed ? -2 : 0;
}

/*
 * Entry point. Layouts: q,k,v,g,dO,o,dq,dk,dv,dg are [S,H,D] (token-major),
 * b and db are [S,H], A_log and dA_log are [H], dt_bias and ddt_bias are
 * [H,D]. S = cu_seqlens[num_seqs]. dO == NULL runs the forward only. o may
 * be NULL when only gradients are wanted. h0 (initial states), hT (final
 * states), dhT (gradient of the final states) and dh0 (gradient of the
 * initial states) are [num_seqs][H][D][V] with rows the key index; each may
 * be NULL (h0 / dhT: zero; hT / dh0: not written). Returns 0 on success, -1
 * on a bad argument, -2 when memory could not be allocated.
 */
int kda_oracle_run(int num_seqs, const int64_t* cu_seqlens, int H, int D,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* b, const double* A_log, const double* dt_bias,
                   double scale, double lower_bound, double eps, const double* dO,
                   double* o, double* dq, double* dk, double* dv, double* dg, double* db,
                   double* dA_log, double* ddt_bias, const double* h0, double* hT,
                   const double* dhT, double* dh0, int num_threads) {
  return oracle_run(num_seqs, cu_seqlens, H, D, q, k, v, g, b, NULL, A_log, dt_bias, scale,
                    lower_bound, eps, dO, o, dq, dk, dv, dg, db, NULL, dA_log, ddt_bias, h0, hT,
                    dhT, dh0, num_threads, 0);
}

/*
 * GDN-2 entry point: the same operator with the scalar beta replaced by a
 * channel-wise erase gate b_t = sigmoid(erase_raw_t) over key channels and a
 * channel-wise write gate w_t = sigmoid(write_raw_t) over value channels
 * ("KDA at the production shape ...", section 1.6 and the section 2.1 op
 * table); see step_cg for the recurrence. erase_raw, write_raw and their
 * gradients derase_raw, dwrite_raw are [S,H,D]; everything else is as in
 * kda_oracle_run.
 */
int gdn2_oracle_run(int num_seqs, const int64_t* cu_seqlens, int H, int D,
                    const double* q, const double* k, const double* v, const double* g,
                    const double* erase_raw, const double* write_raw, const double* A_log,
                    const double* dt_bias, double scale, double lower_bound, double eps,
                    const double* dO, double* o, double* dq, double* dk, double* dv, double* dg,
                    double* derase_raw, double* dwrite_raw, double* dA_log, double* ddt_bias,
                    const double* h0, double* hT, const double* dhT, double* dh0,
                    int num_threads) {
  return oracle_run(num_seqs, cu_seqlens, H, D, q, k, v, g, erase_raw, write_raw, A_log, dt_bias,
                    scale, lower_bound, eps, dO, o, dq, dk, dv, dg, derase_raw, dwrite_raw, dA_log,
                    ddt_bias, h0, hT, dhT, dh0, num_threads, 1);
}
