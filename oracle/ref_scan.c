/*
 * ref_scan.c -- fp64 CPU oracle for the fused selective-scan forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, helper or constant with the CUDA library, and it includes none of it.
 *
 * Sources (page, then section):
 *   [P1] the article at pwwt.cn/news/6372990 on Mamba's hardware-aware
 *        algorithm and parallel associative scan:
 *        s1.1 the discretised recurrence h_t = Abar_t h_{t-1} + Bbar_t x_t,
 *        y_t = C_t h_t + D x_t;  s2.1 an update step as the affine map (a, b)
 *        and the composition rule;  s2.3 padded steps as the identity (1, 0);
 *        s2.4 Abar = exp(delta * A) with A < 0 and delta > 0, fp32 (here fp64)
 *        accumulation;  s3.3 the fused quantities (discretise, b = Bbar x,
 *        scan, C contraction, D residual);  s3.4 per-chunk boundary states;
 *        s4.1 the naive serial loop with a zero initial state.
 *   [P2] "Mamba并行扫描与硬件感知优化：从SSM递推到GPU高效实现"
 *        (bjdmk.com.cn/news/5218626):
 *        s2.2 the operator pair (A_t, b_t) and its merge rule;  s4.2 the
 *        element-wise (diagonal) state transition, states of shape (..., N);
 *        s5.1-s5.2 the Mamba 2 duality (the recurrence as a semiseparable
 *        matrix product, blocks by matrix products and a scan between them).
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes of the repository):
 *   - The transition is diagonal: one scalar decay per (channel d, state n).
 *   - Bbar x is taken as delta * B * x (the pages name zero-order hold but
 *     write no formula for Bbar; delta * B is its first-order form).
 *   - delta is used as given, unless the call asks for the fused step-size
 *     preparation: then the step size is softplus(delta + dt_bias[d]) with
 *     softplus(v) = ln(1 + e^v), optionally clipped to [delta_min, delta_max]
 *     (the pages list softplus and lower/upper clipping of delta among the
 *     fused steps and name a bias on delta; each part is optional).
 *   - The optional gate multiplies the whole output by silu(z) = z / (1+e^-z),
 *     after the D residual is added.
 *   - The state before the first step is h0 when given, else 0.  Steps
 *     t >= valid_len[b] are the identity map (a=1, b=0): the state is frozen
 *     and the output there is exactly 0.
 *   - The chunk boundary state of chunk c is the global state h at step
 *     min((c+1)*chunk_len, L) - 1.
 *
 * Inputs are read as the exact stored values (fp32, or bf16 widened exactly)
 * and widened to double; everything after that is double arithmetic with the
 * C library's exp().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef REF_PLANT
#define REF_PLANT 0 /* >0 only in the mutation tests: plants one known mistake */
#endif

enum { REF_F32 = 0, REF_BF16 = 1 };

/* Exact widening of one stored element to double.  A bf16 value is the upper
 * 16 bits of the fp32 with the same sign, exponent and leading mantissa bits. */
static double ref_load(const void* p, int dtype, int64_t i) {
  if (dtype == REF_F32) return (double)((const float*)p)[i];
  uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* [P1 s2.1], [P2 s2.2]: applying (a1, b1) and then (a2, b2) to h gives
 * a2 (a1 h + b1) + b2, i.e. the pair (a1 a2, a2 b1 + b2).  The b part is
 * order sensitive. */
void ref_combine(double a1, double b1, double a2, double b2, double* a_out, double* b_out) {
#if REF_PLANT == 1
  /* planted mistake: operands of the b part swapped */
  *a_out = a1 * a2;
  *b_out = a1 * b2 + b1;
#else
  *a_out = a1 * a2;
  *b_out = a2 * b1 + b2;
#endif
}

/* [P1 s4.1]: the serial first-order recurrence h_t = a_t h_{t-1} + b_t,
 * starting from h_{-1} = h0.  h[t] receives the state after step t. */
void ref_linear_recurrence(const double* a, const double* b, int64_t L, double h0, double* h) {
  double s = h0;
  for (int64_t t = 0; t < L; ++t) {
    s = a[t] * s + b[t];
    h[t] = s;
  }
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double ref_silu(double z) { return z / (1.0 + exp(-z)); }

/* softplus(v) = ln(1 + e^v), written as max(v, 0) + ln(1 + e^-|v|) so that
 * e^v never overflows. */
static double ref_softplus(double v) {
#if REF_PLANT == 9
  return exp(v); /* planted: exp in place of softplus */
#else
  return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
#endif
}

/*
 * The selective-scan forward over all (b, d) channels.
 *
 * Layouts (row-major, contiguous): x, delta, z, y are [batch, seqlen, dim];
 * B, C are [batch, seqlen, dstate] (shared by every channel d); A is
 * [dim, dstate] fp32; D is [dim] fp32 (NULL = no residual); z NULL = no gate;
 * valid_len is [batch] int32 (NULL = every step valid); h0 is the state before
 * the first step, [batch, dim, dstate] fp32 (NULL = zeros).  y_out receives
 * [batch, seqlen, dim] doubles.  states_out (NULL = not wanted, also when
 * chunk_len <= 0) receives [batch, ceil(seqlen/chunk_len), dim, dstate] doubles;
 * final_out (NULL = not wanted) receives the state after the last step,
 * [batch, dim, dstate] doubles.  The fused step-size preparation: dt_bias
 * ([dim] fp32, NULL = none) is added to delta, delta_softplus != 0 applies
 * softplus to the sum, and delta_clamp != 0 then clips it to
 * [delta_min, delta_max], before delta is used.
 * nthreads <= 0 lets OpenMP choose.  The (b, d) loop is parallel only for
 * speed: each channel is computed by exactly one thread, in program order.
 * Returns 0, or -1 on bad sizes or a failed allocation.
 */
int ref_scan_fwd_full(const void* x, const void* delta, const float* dt_bias, int delta_softplus,
                      int delta_clamp, double delta_min, double delta_max, const float* A, const void* B, const void* C, const float* D,
                      const void* z, const int32_t* valid_len, const float* h0, double* y_out,
                      double* states_out, double* final_out, int64_t batch, int64_t seqlen,
                      int64_t dim, int64_t dstate, int64_t chunk_len, int dtype, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate < 1) return -1;
  if (dtype != REF_F32 && dtype != REF_BF16) return -1;
  const int want_states = (states_out != NULL && chunk_len > 0);
  const int64_t n_chunks = want_states ? (seqlen + chunk_len - 1) / chunk_len : 0;
  const int64_t channels = batch * dim;
  int failed = 0;

#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : failed)
#endif
  for (int64_t bd = 0; bd < channels; ++bd) {
    const int64_t b = bd / dim, d = bd % dim;
    double* h = (double*)malloc((size_t)dstate * sizeof(double));
    if (!h) { failed = 1; continue; }
    for (int64_t n = 0; n < dstate; ++n) /* [P1 s4.1] h_0 = 0 unless given */
      h[n] = h0 ? (double)h0[(b * dim + d) * dstate + n] : 0.0;

    int64_t Lv = seqlen; /* [P1 s2.3] steps from valid_len on are the identity */
    if (valid_len) {
      Lv = valid_len[b];
      if (Lv < 0) Lv = 0;
      if (Lv > seqlen) Lv = seqlen;
    }

    for (int64_t t = 0; t < seqlen; ++t) {
      const int64_t e = (b * seqlen + t) * dim + d; /* element (b, t, d) */
      const int64_t r = (b * seqlen + t) * dstate;  /* row (b, t, :) of B and C */
      double y = 0.0;
      if (t < Lv) {
        double dt = ref_load(delta, dtype, e);
#if REF_PLANT != 8
        if (dt_bias) dt += (double)dt_bias[d]; /* delta + dt_bias[d] */
#endif
        if (delta_softplus) dt = ref_softplus(dt); /* the step size, > 0 */
        if (delta_clamp) dt = dt < delta_min ? delta_min : (dt > delta_max ? delta_max : dt);
        const double xv = ref_load(x, dtype, e);
        double acc = 0.0;
        for (int64_t n = 0; n < dstate; ++n) {
          const double An = (double)A[d * dstate + n];
#if REF_PLANT == 2
          const double a = exp(-dt);                       /* planted: decay without A */
#elif REF_PLANT == 3
          const double a = exp(dt * fabs(An));             /* planted: sign of A lost */
#else
          const double a = exp(dt * An);                   /* [P1 s2.4] Abar = exp(delta A) */
#endif
#if REF_PLANT == 4
          const double bb = ref_load(B, dtype, r + n) * xv; /* planted: delta dropped */
#else
          const double bb = dt * ref_load(B, dtype, r + n) * xv; /* [P1 s3.3] b = Bbar x */
#endif
          h[n] = a * h[n] + bb;                            /* [P1 s1.1] the recurrence */
          acc += ref_load(C, dtype, r + n) * h[n];         /* y = C h */
        }
#if REF_PLANT == 5
        y = acc;                                           /* planted: D residual dropped */
#else
        y = acc + (D ? (double)D[d] * xv : 0.0);           /* [P1 s1.1] + D x */
#endif
        if (z) {
#if REF_PLANT == 6
          y *= ref_silu(xv);                               /* planted: gate on x */
#else
          y *= ref_silu(ref_load(z, dtype, e));            /* gate y * silu(z) */
#endif
        }
      }
      y_out[e] = y;
#if REF_PLANT == 7
      if (want_states && ((t + 2) % chunk_len == 0 || t == seqlen - 1)) { /* planted: off by one */
#else
      if (want_states && ((t + 1) % chunk_len == 0 || t == seqlen - 1)) { /* [P1 s3.4] */
#endif
        double* s = states_out + ((b * n_chunks + t / chunk_len) * dim + d) * dstate;
        for (int64_t n = 0; n < dstate; ++n) s[n] = h[n];
      }
    }
    if (final_out)
      for (int64_t n = 0; n < dstate; ++n) final_out[(b * dim + d) * dstate + n] = h[n];
    free(h);
  }
  return failed ? -1 : 0;
}

/* The forward with delta used as given. */
int ref_scan_fwd_h0(const void* x, const void* delta, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const int32_t* valid_len,
                    const float* h0, double* y_out, double* states_out, double* final_out,
                    int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int64_t chunk_len,
                    int dtype, int nthreads) {
  return ref_scan_fwd_full(x, delta, NULL, 0, 0, 0.0, 0.0, A, B, C, D, z, valid_len, h0, y_out,
                           states_out,
                           final_out, batch, seqlen, dim, dstate, chunk_len, dtype, nthreads);
}

/* The forward from a zero initial state (the call without h0). */
int ref_scan_fwd(const void* x, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const int32_t* valid_len, double* y_out,
                 double* states_out, int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                 int64_t chunk_len, int dtype, int nthreads) {
  return ref_scan_fwd_h0(x, delta, A, B, C, D, z, valid_len, NULL, y_out, states_out, NULL, batch,
                         seqlen, dim, dstate, chunk_len, dtype, nthreads);
}

/* d silu(z) / dz = sigma(z) (1 + z (1 - sigma(z))). */
static double ref_dsilu(double z) {
  const double sg = 1.0 / (1.0 + exp(-z));
  return sg * (1.0 + z * (1.0 - sg));
}

/*
 * The backward of the forward above (delta used as given), for the loss
 * l = sum_{b,t,d} dy[b,t,d] * y[b,t,d]: every gradient of l.  The reverse-mode
 * derivation of the recurrence ([P1] s3.4: the backward replays the chunk
 * boundary states; here every state of the channel is simply kept):
 *   g_t = silu(z_t) (1 without gate), yp_t = sum_n C_tn h_tn + D x_t, y_t = yp_t g_t
 *   dyp_t = dy_t g_t,  dz_t = dy_t yp_t silu'(z_t)
 *   lambda_tn = C_tn dyp_t + a_{t+1,n} lambda_{t+1,n}   (the adjoint of h_t)
 *   with a_t = exp(delta_t A_n), b_t = delta_t B_tn x_t:
 *   d delta_t = sum_n lambda_tn (B_tn x_t + A_n a_tn h_{t-1,n})
 *   d x_t     = sum_n lambda_tn delta_t B_tn + dyp_t D
 *   d B_tn   += lambda_tn delta_t x_t        (summed over d)
 *   d C_tn   += dyp_t h_tn                   (summed over d)
 *   d A_n    += lambda_tn delta_t a_tn h_{t-1,n}   (summed over b, t)
 *   d D      += dyp_t x_t                    (summed over b, t)
 *   d h0_n    = a_{0,n} lambda_{0,n}
 * Steps t >= valid_len contribute nothing (their output is the constant 0
 * and their state update the identity).  dy is [batch, seqlen, dim] doubles;
 * every output is doubles: dx, ddelta, dz [batch, seqlen, dim] (dz NULL
 * without gate), dA [dim, dstate], dB, dC [batch, seqlen, dstate], dD [dim]
 * (NULL = not wanted), dh0 [batch, dim, dstate] (NULL = not wanted).  The
 * summed outputs are overwritten (zeroed first).  Returns 0 or -1.
 */
int ref_scan_bwd(const void* x, const void* delta, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const int32_t* valid_len, const float* h0,
                 const double* dy, double* dx, double* ddelta, double* dA, double* dB,
                 double* dC, double* dD, double* dz, double* dh0, int64_t batch, int64_t seqlen,
                 int64_t dim, int64_t dstate, int dtype, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate < 1) return -1;
  if (dtype != REF_F32 && dtype != REF_BF16) return -1;
  memset(dA, 0, (size_t)(dim * dstate) * sizeof(double));
  memset(dB, 0, (size_t)(batch * seqlen * dstate) * sizeof(double));
  memset(dC, 0, (size_t)(batch * seqlen * dstate) * sizeof(double));
  if (dD) memset(dD, 0, (size_t)dim * sizeof(double));
  const int64_t channels = batch * dim;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : failed)
#endif
  for (int64_t bd = 0; bd < channels; ++bd) {
    const int64_t b = bd / dim, d = bd % dim;
    /* hs[(t + 1) * dstate + n] = h_t, t = -1 .. L-1 */
    double* hs = (double*)malloc((size_t)((seqlen + 1) * dstate) * sizeof(double));
    double* lam = (double*)malloc((size_t)dstate * sizeof(double));
    double* dAl = (double*)calloc((size_t)dstate, sizeof(double));
    if (!hs || !lam || !dAl) { free(hs); free(lam); free(dAl); failed = 1; continue; }
    int64_t Lv = seqlen;
    if (valid_len) {
      Lv = valid_len[b];
      if (Lv < 0) Lv = 0;
      if (Lv > seqlen) Lv = seqlen;
    }
    for (int64_t n = 0; n < dstate; ++n) {
      hs[n] = h0 ? (double)h0[(b * dim + d) * dstate + n] : 0.0;
      lam[n] = 0.0;
    }
    for (int64_t t = 0; t < Lv; ++t) { /* forward, every state kept */
      const int64_t e = (b * seqlen + t) * dim + d, r = (b * seqlen + t) * dstate;
      const double dt = ref_load(delta, dtype, e), xv = ref_load(x, dtype, e);
      for (int64_t n = 0; n < dstate; ++n)
        hs[(t + 1) * dstate + n] = exp(dt * (double)A[d * dstate + n]) * hs[t * dstate + n] +
                                   dt * ref_load(B, dtype, r + n) * xv;
    }
    double dDl = 0.0;
    for (int64_t t = seqlen - 1; t >= 0; --t) {
      const int64_t e = (b * seqlen + t) * dim + d, r = (b * seqlen + t) * dstate;
      if (t >= Lv) {
        dx[e] = 0.0; ddelta[e] = 0.0;
        if (dz) dz[e] = 0.0;
        continue;
      }
      const double dt = ref_load(delta, dtype, e), xv = ref_load(x, dtype, e);
      const double Dd = D ? (double)D[d] : 0.0;
      double yp = Dd * xv;
      for (int64_t n = 0; n < dstate; ++n) yp += ref_load(C, dtype, r + n) * hs[(t + 1) * dstate + n];
      double g = 1.0;
      if (z) {
        const double zv = ref_load(z, dtype, e);
        g = ref_silu(zv);
#if REF_PLANT == 12
        dz[e] = dy[e] * yp * g; /* planted: silu in place of its derivative */
#else
        dz[e] = dy[e] * yp * ref_dsilu(zv);
#endif
      }
      const double dyp = dy[e] * g;
      double ddt = 0.0, dxv = dyp * Dd;
      dDl += dyp * xv;
      for (int64_t n = 0; n < dstate; ++n) {
        const double An = (double)A[d * dstate + n];
        const double a = exp(dt * An), Bn = ref_load(B, dtype, r + n);
        const double hp = hs[t * dstate + n]; /* h_{t-1} */
        lam[n] += ref_load(C, dtype, r + n) * dyp;
        ddt += lam[n] * (Bn * xv + An * a * hp);
        dxv += lam[n] * dt * Bn;
#ifdef _OPENMP
#pragma omp atomic
#endif
        dB[r + n] += lam[n] * dt * xv;
#ifdef _OPENMP
#pragma omp atomic
#endif
        dC[r + n] += dyp * hs[(t + 1) * dstate + n];
#if REF_PLANT == 11
        dAl[n] += lam[n] * a * hp; /* planted: delta factor of dA lost */
#else
        dAl[n] += lam[n] * dt * a * hp;
#endif
#if REF_PLANT == 10
        lam[n] *= exp((t + 1 < Lv ? ref_load(delta, dtype, e + dim) : dt) * An); /* planted: a_{t+1} */
#else
        lam[n] *= a; /* carry to step t-1: a_t lambda_t */
#endif
      }
      ddelta[e] = ddt;
      dx[e] = dxv;
    }
    for (int64_t n = 0; n < dstate; ++n) {
#ifdef _OPENMP
#pragma omp atomic
#endif
      dA[d * dstate + n] += dAl[n];
      if (dh0) dh0[(b * dim + d) * dstate + n] = lam[n];
    }
    if (dD) {
#ifdef _OPENMP
#pragma omp atomic
#endif
      dD[d] += dDl;
    }
    free(hs); free(lam); free(dAl);
  }
  return failed ? -1 : 0;
}

/*
 * The state-space-duality (SSD) form of the scan ([P2] s5.1-s5.2, the Mamba 2
 * section): the same linear recurrence, with one decay per head shared by all
 * of the head's channels and states, which is what lets the in-block work be
 * written as matrix products.  Channels are grouped in nheads heads of
 * headdim channels (d = h * headdim + p); per head h the step size delta is
 * one value per (b, t, h) and A is one scalar A[h] < 0.  For every (b, h, p)
 * and state n, from h_{-1} = h0 (else 0):
 *   a_t = exp(delta_{b,t,h} A_h),  h_tn = a_t h_{t-1,n} + delta_{b,t,h} B_{b,t,n} x_{b,t,d}
 *   y_{b,t,d} = (sum_n C_{b,t,n} h_tn + D_d x_{b,t,d}) * silu(z_{b,t,d})   (gate optional)
 * Steps t >= valid_len[b] are the identity and their output is exactly 0, as
 * in the scan above.  This is the definition; the blocked matrix form that a
 * fast implementation uses is checked against it by the tests (the quadratic
 * form y = M x with M[t,s] = (C_t . B_s) exp(A_h sum_{s<r<=t} delta_r) delta_s).
 * Layouts: x, z [batch, seqlen, nheads*headdim]; delta [batch, seqlen, nheads];
 * A [nheads] fp32; B, C [batch, seqlen, dstate]; D [nheads*headdim] fp32 or
 * NULL; h0 and final [batch, nheads*headdim, dstate] (fp32 in, double out, NULL
 * = zero / not wanted); y_out [batch, seqlen, nheads*headdim] doubles.
 */
int ref_ssd_fwd(const void* x, const void* delta, const float* A, const void* B, const void* C,
                const float* D, const void* z, const int32_t* valid_len, const float* h0,
                double* y_out, double* final_out, int64_t batch, int64_t seqlen, int64_t nheads,
                int64_t headdim, int64_t dstate, int dtype, int nthreads) {
  if (batch < 0 || seqlen < 0 || nheads < 0 || headdim < 1 || dstate < 1) return -1;
  if (dtype != REF_F32 && dtype != REF_BF16) return -1;
  const int64_t dim = nheads * headdim, channels = batch * dim;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : failed)
#endif
  for (int64_t bd = 0; bd < channels; ++bd) {
    const int64_t b = bd / dim, d = bd % dim, hd = d / headdim;
    double* h = (double*)malloc((size_t)dstate * sizeof(double));
    if (!h) { failed = 1; continue; }
    for (int64_t n = 0; n < dstate; ++n) h[n] = h0 ? (double)h0[(b * dim + d) * dstate + n] : 0.0;
    int64_t Lv = seqlen;
    if (valid_len) {
      Lv = valid_len[b];
      if (Lv < 0) Lv = 0;
      if (Lv > seqlen) Lv = seqlen;
    }
    const double Ah = (double)A[hd];
    for (int64_t t = 0; t < seqlen; ++t) {
      const int64_t e = (b * seqlen + t) * dim + d;
      const int64_t r = (b * seqlen + t) * dstate;
      double y = 0.0;
      if (t < Lv) {
        const double dt = ref_load(delta, dtype, (b * seqlen + t) * nheads + hd);
#if REF_PLANT == 13
        const double xv = ref_load(x, dtype, (b * seqlen + t) * dim + d % headdim); /* planted: head offset lost */
#else
        const double xv = ref_load(x, dtype, e);
#endif
        const double a = exp(dt * Ah); /* one decay for the whole head */
        double acc = 0.0;
        for (int64_t n = 0; n < dstate; ++n) {
#if REF_PLANT == 14
          h[n] = a * (h[n] + dt * ref_load(B, dtype, r + n) * xv); /* planted: input decayed too */
#else
          h[n] = a * h[n] + dt * ref_load(B, dtype, r + n) * xv;
#endif
          acc += ref_load(C, dtype, r + n) * h[n];
        }
        y = acc + (D ? (double)D[d] * xv : 0.0);
        if (z) y *= ref_silu(ref_load(z, dtype, e));
      }
      y_out[e] = y;
    }
    if (final_out)
      for (int64_t n = 0; n < dstate; ++n) final_out[(b * dim + d) * dstate + n] = h[n];
    free(h);
  }
  return failed ? -1 : 0;
}

/* Version tag so a loader can tell which oracle build (plain or planted) it has. */
int ref_plant_id(void) { return REF_PLANT; }
