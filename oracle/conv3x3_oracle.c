/*
 * conv3x3_oracle.c -- the plain, slow, obviously correct CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes.  The subject page ("UNet diffusion in C++/CUDA" by clu0,
 * sourcepulse.org project page, sections "How It Works" and "Highlighted
 * Details") describes custom 3x3 convolution kernels, forward and backward,
 * inside a UNet that aims to match PyTorch.  The page never writes the
 * convolution down, so this file follows the textbook / PyTorch Conv2d
 * definition of a stride-1, zero-pad-1, dilation-1, groups-1 3x3
 * cross-correlation (no kernel flip):
 *
 *   forward  z[n,h,w,k] = b[k] + sum_{r,s,c} x[n,h+r-1,w+s-1,c] * wt[k,r,s,c]
 *            y = z                         (act = 0)
 *            y = z * sigmoid(z)            (act = 1, SiLU)
 *            y = z >= 0 ? z : 0.2 z        (act = 2, bias + leaky ReLU: the fused
 *                                           bias + activation op of the StyleGAN2
 *                                           custom-kernel blog, page titled "Dim3
 *                                           grid calculation code", opening
 *                                           paragraphs; it gives no slope or
 *                                           gain, so slope 0.2 and no gain)
 *   dgrad   dx[n,h,w,c] = sum_{r,s,k} dz[n,h+1-r,w+1-s,k] * wt[k,r,s,c]
 *   dgrad through the input's activation, x = act(zin):
 *           dzin[n,h,w,c] = act'(zin[n,h,w,c]) * dx[n,h,w,c]
 *   wgrad   dw[k,r,s,c] = sum_{n,h,w} dz[n,h,w,k] * x[n,h+r-1,w+s-1,c]
 *   dbias   db[k]       = sum_{n,h,w} dz[n,h,w,k]
 *
 * Out-of-range taps contribute zero.  Layouts: activations NHWC (c fastest),
 * weights KRSC = [Cout][3][3][Cin] (c fastest).  All arithmetic is IEEE
 * double; inputs arrive already widened from their stored precision.
 *
 * Parallelism is plain pthreads over the outermost independent loop; each
 * output element is still summed in the single fixed order written below, so
 * results do not depend on the thread count.
 *
 * Parity pins: every function here is pinned by the CPU tests (centre and
 * off-centre deltas, the all-ones border pattern, the 1x1 GEMM special case,
 * the adjoint and bilinear identities, finite differences, an explicit
 * im2col brute force, a hand-computed fixture and torch's float64 conv2d).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_MAX_THREADS 256

static int g_threads = 0; /* 0 = all online cores */

void oracle_set_threads(int n) { g_threads = n < 0 ? 0 : n; }

int oracle_get_threads(void) {
  if (g_threads > 0) return g_threads > ORACLE_MAX_THREADS ? ORACLE_MAX_THREADS : g_threads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  if (n < 1) n = 1;
  if (n > ORACLE_MAX_THREADS) n = ORACLE_MAX_THREADS;
  return (int)n;
}

/* ---- a minimal parallel-for: items [0, count) split into contiguous slices ---- */
typedef void (*item_fn)(void* ctx, int64_t item);
typedef struct { item_fn fn; void* ctx; int64_t lo, hi; } slice_t;

static void* run_slice(void* p) {
  slice_t* s = (slice_t*)p;
  for (int64_t i = s->lo; i < s->hi; ++i) s->fn(s->ctx, i);
  return NULL;
}

static void parallel_for(int64_t count, item_fn fn, void* ctx) {
  int nt = oracle_get_threads();
  if (nt > count) nt = (int)(count > 0 ? count : 1);
  if (nt <= 1) {
    for (int64_t i = 0; i < count; ++i) fn(ctx, i);
    return;
  }
  pthread_t th[ORACLE_MAX_THREADS];
  slice_t sl[ORACLE_MAX_THREADS];
  int started[ORACLE_MAX_THREADS];
  for (int t = 0; t < nt; ++t) {
    sl[t].fn = fn;
    sl[t].ctx = ctx;
    sl[t].lo = count * t / nt;
    sl[t].hi = count * (t + 1) / nt;
    started[t] = pthread_create(&th[t], NULL, run_slice, &sl[t]) == 0;
    if (!started[t]) run_slice(&sl[t]); /* could not spawn: do it inline */
  }
  for (int t = 0; t < nt; ++t)
    if (started[t]) pthread_join(th[t], NULL);
}

typedef struct {
  const double *x, *wt, *bias, *dz;
  double *out, *out2;
  int64_t N, Cin, Cout, H, W;
  int act;
  const int64_t* idx;
  const double* zin; /* dgrad through an activation: its pre-activation input */
  int64_t u;         /* strided convolution: stride (output Ho = (H-1)/u + 1, Wo likewise) */
} job_t;

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^{-z}).  For very negative z, e^{-z}
 * overflows to +inf and the quotient is -0, the correct limit. */
double oracle_silu_f64(double z) { return z / (1.0 + exp(-z)); }

/* leaky ReLU with negative slope 0.2 */
double oracle_lrelu_f64(double z) { return z >= 0.0 ? z : 0.2 * z; }

static double apply_act(int act, double z) {
  if (act == 1) return oracle_silu_f64(z);
  if (act == 2) return oracle_lrelu_f64(z);
  return z;
}

/* Derivative of the activation at z.
 *   SiLU:       d/dz [z s(z)] = s(z) + z s(z)(1 - s(z)) = s(z) (1 + z (1 - s(z))),
 *               s the logistic sigmoid.
 *   leaky ReLU: 1 for z > 0 and 0.2 otherwise; at z = 0 both one-sided
 *               derivatives exist and the lower one is taken, as PyTorch's
 *               leaky_relu backward does.
 *   none:       1. */
double oracle_act_grad_f64(int act, double z) {
  if (act == 1) {
    double sg = 1.0 / (1.0 + exp(-z));
    return sg * (1.0 + z * (1.0 - sg));
  }
  if (act == 2) return z > 0.0 ? 1.0 : 0.2;
  return 1.0;
}

/* ---------------- forward ---------------- */
static double fwd_point(const job_t* j, int64_t n, int64_t h, int64_t w, int64_t k) {
  double acc = j->bias ? j->bias[k] : 0.0;
  for (int64_t r = 0; r < 3; ++r) {
    int64_t hh = h + r - 1;
    if (hh < 0 || hh >= j->H) continue;
    for (int64_t s = 0; s < 3; ++s) {
      int64_t ww = w + s - 1;
      if (ww < 0 || ww >= j->W) continue;
      const double* xp = j->x + ((n * j->H + hh) * j->W + ww) * j->Cin;
      const double* wp = j->wt + ((k * 3 + r) * 3 + s) * j->Cin;
      for (int64_t c = 0; c < j->Cin; ++c) acc += xp[c] * wp[c];
    }
  }
  return apply_act(j->act, acc);
}

static void fwd_row(void* ctx, int64_t nh) { /* one (n, h) output row */
  const job_t* j = (const job_t*)ctx;
  int64_t n = nh / j->H, h = nh % j->H;
  for (int64_t w = 0; w < j->W; ++w)
    for (int64_t k = 0; k < j->Cout; ++k)
      j->out[((n * j->H + h) * j->W + w) * j->Cout + k] = fwd_point(j, n, h, w, k);
}

void oracle_conv3x3_fwd_f64(const double* x, const double* wt, const double* bias, double* y,
                            int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W, int act) {
  job_t j = {x, wt, bias, NULL, y, NULL, N, Cin, Cout, H, W, act, NULL};
  parallel_for(N * H, fwd_row, &j);
}

/* sampled forward: out[i] = y at linear NHWC index idx[i] */
static void fwd_at_item(void* ctx, int64_t i) {
  const job_t* j = (const job_t*)ctx;
  int64_t e = j->idx[i];
  int64_t k = e % j->Cout, p = e / j->Cout;
  int64_t w = p % j->W, h = (p / j->W) % j->H, n = p / (j->W * j->H);
  j->out[i] = fwd_point(j, n, h, w, k);
}

void oracle_conv3x3_fwd_at_f64(const double* x, const double* wt, const double* bias,
                               int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W, int act,
                               const int64_t* idx, int64_t count, double* out) {
  job_t j = {x, wt, bias, NULL, out, NULL, N, Cin, Cout, H, W, act, idx};
  parallel_for(count, fwd_at_item, &j);
}

/* ---------------- dgrad ---------------- */
static double dgrad_point(const job_t* j, int64_t n, int64_t h, int64_t w, int64_t c) {
  double acc = 0.0;
  for (int64_t r = 0; r < 3; ++r) {
    int64_t hh = h + 1 - r;
    if (hh < 0 || hh >= j->H) continue;
    for (int64_t s = 0; s < 3; ++s) {
      int64_t ww = w + 1 - s;
      if (ww < 0 || ww >= j->W) continue;
      const double* dzp = j->dz + ((n * j->H + hh) * j->W + ww) * j->Cout;
      for (int64_t k = 0; k < j->Cout; ++k)
        acc += dzp[k] * j->wt[((k * 3 + r) * 3 + s) * j->Cin + c];
    }
  }
  return acc;
}

static void dgrad_row(void* ctx, int64_t nh) {
  const job_t* j = (const job_t*)ctx;
  int64_t n = nh / j->H, h = nh % j->H;
  for (int64_t w = 0; w < j->W; ++w)
    for (int64_t c = 0; c < j->Cin; ++c)
      j->out[((n * j->H + h) * j->W + w) * j->Cin + c] = dgrad_point(j, n, h, w, c);
}

void oracle_conv3x3_dgrad_f64(const double* dz, const double* wt, double* dx,
                              int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W) {
  job_t j = {NULL, wt, NULL, dz, dx, NULL, N, Cin, Cout, H, W, 0, NULL};
  parallel_for(N * H, dgrad_row, &j);
}

static void dgrad_at_item(void* ctx, int64_t i) {
  const job_t* j = (const job_t*)ctx;
  int64_t e = j->idx[i];
  int64_t c = e % j->Cin, p = e / j->Cin;
  int64_t w = p % j->W, h = (p / j->W) % j->H, n = p / (j->W * j->H);
  j->out[i] = dgrad_point(j, n, h, w, c);
}

void oracle_conv3x3_dgrad_at_f64(const double* dz, const double* wt,
                                 int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W,
                                 const int64_t* idx, int64_t count, double* out) {
  job_t j = {NULL, wt, NULL, dz, out, NULL, N, Cin, Cout, H, W, 0, idx};
  parallel_for(count, dgrad_at_item, &j);
}

/* ---------------- dgrad through the previous layer's activation ----------------
 * When this convolution's input is x = act(zin), the chain rule gives the
 * gradient with respect to zin as
 *   dzin[n,h,w,c] = act'(zin[n,h,w,c]) * dx[n,h,w,c],
 * dx the plain dgrad above; zin has the layout of dx. */
static void dgrad_act_row(void* ctx, int64_t nh) {
  const job_t* j = (const job_t*)ctx;
  int64_t n = nh / j->H, h = nh % j->H;
  for (int64_t w = 0; w < j->W; ++w)
    for (int64_t c = 0; c < j->Cin; ++c) {
      int64_t e = ((n * j->H + h) * j->W + w) * j->Cin + c;
      j->out[e] = oracle_act_grad_f64(j->act, j->zin[e]) * dgrad_point(j, n, h, w, c);
    }
}

void oracle_conv3x3_dgrad_act_f64(const double* dz, const double* wt, const double* zin, int act,
                                  double* dx, int64_t N, int64_t Cin, int64_t Cout, int64_t H,
                                  int64_t W) {
  job_t j = {NULL, wt, NULL, dz, dx, NULL, N, Cin, Cout, H, W, act, NULL, zin};
  parallel_for(N * H, dgrad_act_row, &j);
}

static void dgrad_act_at_item(void* ctx, int64_t i) {
  const job_t* j = (const job_t*)ctx;
  int64_t e = j->idx[i];
  int64_t c = e % j->Cin, p = e / j->Cin;
  int64_t w = p % j->W, h = (p / j->W) % j->H, n = p / (j->W * j->H);
  j->out[i] = oracle_act_grad_f64(j->act, j->zin[e]) * dgrad_point(j, n, h, w, c);
}

void oracle_conv3x3_dgrad_act_at_f64(const double* dz, const double* wt, const double* zin, int act,
                                     int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W,
                                     const int64_t* idx, int64_t count, double* out) {
  job_t j = {NULL, wt, NULL, dz, out, NULL, N, Cin, Cout, H, W, act, idx, zin};
  parallel_for(count, dgrad_act_at_item, &j);
}

/* ---------------- wgrad + dbias ---------------- */
/* One output channel k: the full [3][3][Cin] slab of dw and db[k]; the sum over
 * pixels runs in increasing (n, h, w) order for every element. */
static void wgrad_k(void* ctx, int64_t k) {
  const job_t* j = (const job_t*)ctx;
  double* dwk = j->out + k * 9 * j->Cin;
  for (int64_t e = 0; e < 9 * j->Cin; ++e) dwk[e] = 0.0;
  double db = 0.0;
  for (int64_t n = 0; n < j->N; ++n)
    for (int64_t h = 0; h < j->H; ++h)
      for (int64_t w = 0; w < j->W; ++w) {
        double d = j->dz[((n * j->H + h) * j->W + w) * j->Cout + k];
        db += d;
        for (int64_t r = 0; r < 3; ++r) {
          int64_t hh = h + r - 1;
          if (hh < 0 || hh >= j->H) continue;
          for (int64_t s = 0; s < 3; ++s) {
            int64_t ww = w + s - 1;
            if (ww < 0 || ww >= j->W) continue;
            const double* xp = j->x + ((n * j->H + hh) * j->W + ww) * j->Cin;
            double* acc = dwk + (r * 3 + s) * j->Cin;
            for (int64_t c = 0; c < j->Cin; ++c) acc[c] += d * xp[c];
          }
        }
      }
  if (j->out2) j->out2[k] = db;
}

void oracle_conv3x3_wgrad_f64(const double* x, const double* dz, double* dw, double* db,
                              int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W) {
  job_t j = {x, NULL, NULL, dz, dw, db, N, Cin, Cout, H, W, 0, NULL};
  parallel_for(Cout, wgrad_k, &j);
}

/* sampled wgrad: out[i] = dw at linear KRSC index idx[i] */
static void wgrad_at_item(void* ctx, int64_t i) {
  const job_t* j = (const job_t*)ctx;
  int64_t e = j->idx[i];
  int64_t c = e % j->Cin, rs = (e / j->Cin) % 9, k = e / (9 * j->Cin);
  int64_t r = rs / 3, s = rs % 3;
  double acc = 0.0;
  for (int64_t n = 0; n < j->N; ++n)
    for (int64_t h = 0; h < j->H; ++h) {
      int64_t hh = h + r - 1;
      if (hh < 0 || hh >= j->H) continue;
      for (int64_t w = 0; w < j->W; ++w) {
        int64_t ww = w + s - 1;
        if (ww < 0 || ww >= j->W) continue;
        acc += j->dz[((n * j->H + h) * j->W + w) * j->Cout + k] *
               j->x[((n * j->H + hh) * j->W + ww) * j->Cin + c];
      }
    }
  j->out[i] = acc;
}

void oracle_conv3x3_wgrad_at_f64(const double* x, const double* dz,
                                 int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W,
                                 const int64_t* idx, int64_t count, double* out) {
  job_t j = {x, NULL, NULL, dz, out, NULL, N, Cin, Cout, H, W, 0, idx};
  parallel_for(count, wgrad_at_item, &j);
}

static void dbias_k(void* ctx, int64_t k) {
  const job_t* j = (const job_t*)ctx;
  double acc = 0.0;
  int64_t P = j->N * j->H * j->W;
  for (int64_t p = 0; p < P; ++p) acc += j->dz[p * j->Cout + k];
  j->out[k] = acc;
}

void oracle_conv3x3_dbias_f64(const double* dz, double* db, int64_t N, int64_t Cout, int64_t H,
                              int64_t W) {
  job_t j = {NULL, NULL, NULL, dz, db, NULL, N, 0, Cout, H, W, 0, NULL};
  parallel_for(Cout, dbias_k, &j);
}

/* ---------------- strided convolution (stride u, zero padding 1) ----------------
 * A UNet's downsampling conv: the same 3x3 window, moved u pixels at a time.
 *   Ho = (H - 1) / u + 1,  Wo = (W - 1) / u + 1
 *   forward  z[n,ho,wo,k] = b[k] + sum_{r,s,c} x[n, u ho + r - 1, u wo + s - 1, c] wt[k,r,s,c]
 *            y = act(z)
 *   dgrad    dx[n,h,w,c] = sum over (ho, wo, r, s) with u ho + r - 1 = h and
 *            u wo + s - 1 = w of dz[n,ho,wo,k] wt[k,r,s,c]   (the adjoint of the forward)
 *   wgrad    dw[k,r,s,c] = sum_{n,ho,wo} dz[n,ho,wo,k] x[n, u ho + r - 1, u wo + s - 1, c]
 *   dbias    db[k]       = sum_{n,ho,wo} dz[n,ho,wo,k]
 * x, dx: [N][H][W][Cin]; y, dz: [N][Ho][Wo][Cout]; out-of-range taps contribute zero. */
static int64_t s_out(int64_t len, int64_t u) { return (len - 1) / u + 1; }

static double sfwd_point(const job_t* j, int64_t n, int64_t ho, int64_t wo, int64_t k) {
  double acc = j->bias ? j->bias[k] : 0.0;
  for (int64_t r = 0; r < 3; ++r) {
    int64_t hh = j->u * ho + r - 1;
    if (hh < 0 || hh >= j->H) continue;
    for (int64_t s = 0; s < 3; ++s) {
      int64_t ww = j->u * wo + s - 1;
      if (ww < 0 || ww >= j->W) continue;
      const double* xp = j->x + ((n * j->H + hh) * j->W + ww) * j->Cin;
      const double* wp = j->wt + ((k * 3 + r) * 3 + s) * j->Cin;
      for (int64_t c = 0; c < j->Cin; ++c) acc += xp[c] * wp[c];
    }
  }
  return apply_act(j->act, acc);
}

static void sfwd_item(void* ctx, int64_t i) { /* one output element, linear [N][Ho][Wo][Cout] index */
  const job_t* j = (const job_t*)ctx;
  const int64_t Ho = s_out(j->H, j->u), Wo = s_out(j->W, j->u);
  int64_t e = j->idx ? j->idx[i] : i;
  int64_t k = e % j->Cout, p = e / j->Cout;
  int64_t wo = p % Wo, ho = (p / Wo) % Ho, n = p / (Wo * Ho);
  j->out[i] = sfwd_point(j, n, ho, wo, k);
}

void oracle_conv3x3_fwd_strided_f64(const double* x, const double* wt, const double* bias,
                                    double* y, int64_t N, int64_t Cin, int64_t Cout, int64_t H,
                                    int64_t W, int64_t u, int act) {
  job_t j = {x, wt, bias, NULL, y, NULL, N, Cin, Cout, H, W, act, NULL, NULL, u};
  parallel_for(N * s_out(H, u) * s_out(W, u) * Cout, sfwd_item, &j);
}

void oracle_conv3x3_fwd_strided_at_f64(const double* x, const double* wt, const double* bias,
                                       int64_t N, int64_t Cin, int64_t Cout, int64_t H, int64_t W,
                                       int64_t u, int act, const int64_t* idx, int64_t count,
                                       double* out) {
  job_t j = {x, wt, bias, NULL, out, NULL, N, Cin, Cout, H, W, act, idx, NULL, u};
  parallel_for(count, sfwd_item, &j);
}

static double sdgrad_point(const job_t* j, int64_t n, int64_t h, int64_t w, int64_t c) {
  const int64_t Ho = s_out(j->H, j->u), Wo = s_out(j->W, j->u);
  double acc = 0.0;
  for (int64_t r = 0; r < 3; ++r) {
    int64_t th = h + 1 - r; /* = u ho */
    if (th < 0 || th % j->u != 0 || th / j->u >= Ho) continue;
    int64_t ho = th / j->u;
    for (int64_t s = 0; s < 3; ++s) {
      int64_t tw = w + 1 - s; /* = u wo */
      if (tw < 0 || tw % j->u != 0 || tw / j->u >= Wo) continue;
      int64_t wo = tw / j->u;
      const double* dzp = j->dz + ((n * Ho + ho) * Wo + wo) * j->Cout;
      for (int64_t k = 0; k < j->Cout; ++k)
        acc += dzp[k] * j->wt[((k * 3 + r) * 3 + s) * j->Cin + c];
    }
  }
  return acc;
}

static void sdgrad_item(void* ctx, int64_t i) { /* one element of dx, linear [N][H][W][Cin] index */
  const job_t* j = (const job_t*)ctx;
  int64_t e = j->idx ? j->idx[i] : i;
  int64_t c = e % j->Cin, p = e / j->Cin;
  int64_t w = p % j->W, h = (p / j->W) % j->H, n = p / (j->W * j->H);
  j->out[i] = sdgrad_point(j, n, h, w, c);
}

void oracle_conv3x3_dgrad_strided_f64(const double* dz, const double* wt, double* dx, int64_t N,
                                      int64_t Cin, int64_t Cout, int64_t H, int64_t W, int64_t u) {
  job_t j = {NULL, wt, NULL, dz, dx, NULL, N, Cin, Cout, H, W, 0, NULL, NULL, u};
  parallel_for(N * H * W * Cin, sdgrad_item, &j);
}

void oracle_conv3x3_dgrad_strided_at_f64(const double* dz, const double* wt, int64_t N,
                                         int64_t Cin, int64_t Cout, int64_t H, int64_t W,
                                         int64_t u, const int64_t* idx, int64_t count,
                                         double* out) {
  job_t j = {NULL, wt, NULL, dz, out, NULL, N, Cin, Cout, H, W, 0, idx, NULL, u};
  parallel_for(count, sdgrad_item, &j);
}

/* one element of dw (linear KRSC index), or db[k] when the index is 9*Cin*Cout + k;
 * the pixel sum runs in increasing (n, ho, wo) order */
static void swgrad_item(void* ctx, int64_t i) {
  const job_t* j = (const job_t*)ctx;
  const int64_t Ho = s_out(j->H, j->u), Wo = s_out(j->W, j->u);
  int64_t e = j->idx ? j->idx[i] : i;
  double acc = 0.0;
  if (e >= 9 * j->Cin * j->Cout) {
    int64_t k = e - 9 * j->Cin * j->Cout;
    for (int64_t p = 0; p < j->N * Ho * Wo; ++p) acc += j->dz[p * j->Cout + k];
    j->out[i] = acc;
    return;
  }
  int64_t c = e % j->Cin, rs = (e / j->Cin) % 9, k = e / (9 * j->Cin);
  int64_t r = rs / 3, s = rs % 3;
  for (int64_t n = 0; n < j->N; ++n)
    for (int64_t ho = 0; ho < Ho; ++ho) {
      int64_t hh = j->u * ho + r - 1;
      if (hh < 0 || hh >= j->H) continue;
      for (int64_t wo = 0; wo < Wo; ++wo) {
        int64_t ww = j->u * wo + s - 1;
        if (ww < 0 || ww >= j->W) continue;
        acc += j->dz[((n * Ho + ho) * Wo + wo) * j->Cout + k] *
               j->x[((n * j->H + hh) * j->W + ww) * j->Cin + c];
      }
    }
  j->out[i] = acc;
}

/* dwdb: 9*Cin*Cout dw values (KRSC) followed by Cout db values */
void oracle_conv3x3_wgrad_strided_f64(const double* x, const double* dz, double* dwdb, int64_t N,
                                      int64_t Cin, int64_t Cout, int64_t H, int64_t W, int64_t u) {
  job_t j = {x, NULL, NULL, dz, dwdb, NULL, N, Cin, Cout, H, W, 0, NULL, NULL, u};
  parallel_for(9 * Cin * Cout + Cout, swgrad_item, &j);
}

void oracle_conv3x3_wgrad_strided_at_f64(const double* x, const double* dz, int64_t N,
                                         int64_t Cin, int64_t Cout, int64_t H, int64_t W,
                                         int64_t u, const int64_t* idx, int64_t count,
                                         double* out) {
  job_t j = {x, NULL, NULL, dz, out, NULL, N, Cin, Cout, H, W, 0, idx, NULL, u};
  parallel_for(count, swgrad_item, &j);
}
