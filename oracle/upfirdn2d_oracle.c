/*
 * upfirdn2d_oracle.c -- TEST INFRASTRUCTURE ONLY: the plain CPU definition of
 * upfirdn2d that the GPU kernel is checked against.  Loaded by tests/,
 * __graft_entry__.smoke() and bench.py's CPU-baseline leg only; never by the
 * product path.  Shares no code with the CUDA library.
 *
 * The operation is the one the StyleGAN2 custom-kernel blog (page titled
 * "Dim3 grid calculation code", first paragraph) describes for filtered
 * up/downsampling: every channel of every image goes through four steps, in
 * this order,
 *   1. upsample: insert (up - 1) zeros after each pixel, along both axes;
 *   2. pad: add pad_y0 / pad_y1 zero rows above / below and pad_x0 / pad_x1
 *      zero columns left / right;
 *   3. FIR filter: 2-D convolution with the kh x kw kernel f, keeping the
 *      positions where the kernel lies wholly inside the padded plane;
 *   4. downsample: keep every down-th pixel, starting with the first.
 * Readings where the page is silent (its kernel formula did not survive the
 * extraction): "convolution" is taken literally, with the kernel flipped
 *   F[m][l] = sum_{a,b} f[a][b] * Pd[m + kh - 1 - a][l + kw - 1 - b],
 * pads are non-negative (zeros only, no cropping), and the output size is
 *   Ho = (H * up + pad_y0 + pad_y1 - kh) / down + 1   (likewise Wo).
 * Layout: x [N][H][W][C], y [N][Ho][Wo][C] (channels fastest), f [kh][kw].
 *
 * Arithmetic in double; each output is one fixed-order sum.  pthreads over the
 * N * C independent planes.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

int oracle_get_threads(void);

typedef struct {
  const double* x;
  const double* f;
  double* y;
  int64_t N, H, W, C, up, down, px0, px1, py0, py1, kh, kw;
  const int64_t* idx;
} ufd_job_t;

typedef void (*ufd_item_fn)(void* ctx, int64_t item);
typedef struct {
  ufd_item_fn fn;
  void* ctx;
  int64_t begin, end;
} ufd_slice_t;

static void* ufd_run_slice(void* p) {
  ufd_slice_t* s = (ufd_slice_t*)p;
  for (int64_t i = s->begin; i < s->end; ++i) s->fn(s->ctx, i);
  return NULL;
}

static void ufd_parallel_for(int64_t count, ufd_item_fn fn, void* ctx) {
  int nt = oracle_get_threads();
  if (nt > count) nt = (int)count;
  if (nt <= 1) {
    for (int64_t i = 0; i < count; ++i) fn(ctx, i);
    return;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
  ufd_slice_t* sl = (ufd_slice_t*)malloc(sizeof(ufd_slice_t) * nt);
  for (int t = 0; t < nt; ++t) {
    sl[t].fn = fn;
    sl[t].ctx = ctx;
    sl[t].begin = count * t / nt;
    sl[t].end = count * (t + 1) / nt;
    pthread_create(&th[t], NULL, ufd_run_slice, &sl[t]);
  }
  for (int t = 0; t < nt; ++t) pthread_join(th[t], NULL);
  free(th);
  free(sl);
}

int64_t oracle_upfirdn2d_out_len(int64_t len, int64_t up, int64_t down, int64_t p0, int64_t p1,
                                 int64_t k) {
  int64_t full = len * up + p0 + p1 - k;
  return full < 0 ? 0 : full / down + 1;
}

/* One (image, channel) plane through the four steps, each materialised. */
static void ufd_plane(void* ctx, int64_t nc) {
  const ufd_job_t* j = (const ufd_job_t*)ctx;
  const int64_t n = nc / j->C, c = nc % j->C;
  /* 1. upsample: zeros after each pixel */
  const int64_t Hu = j->H * j->up, Wu = j->W * j->up;
  double* u = (double*)calloc((size_t)(Hu * Wu), sizeof(double));
  for (int64_t h = 0; h < j->H; ++h)
    for (int64_t w = 0; w < j->W; ++w)
      u[(h * j->up) * Wu + w * j->up] = j->x[((n * j->H + h) * j->W + w) * j->C + c];
  /* 2. pad with zeros on each side */
  const int64_t Hp = Hu + j->py0 + j->py1, Wp = Wu + j->px0 + j->px1;
  double* pd = (double*)calloc((size_t)(Hp * Wp), sizeof(double));
  for (int64_t h = 0; h < Hu; ++h)
    for (int64_t w = 0; w < Wu; ++w) pd[(h + j->py0) * Wp + (w + j->px0)] = u[h * Wu + w];
  /* 3. FIR filter: convolution with f over the positions where it fits */
  const int64_t Hf = Hp - j->kh + 1, Wf = Wp - j->kw + 1;
  double* fl = (double*)calloc((size_t)(Hf > 0 && Wf > 0 ? Hf * Wf : 1), sizeof(double));
  for (int64_t m = 0; m < Hf; ++m)
    for (int64_t l = 0; l < Wf; ++l) {
      double acc = 0.0;
      for (int64_t a = 0; a < j->kh; ++a)
        for (int64_t b = 0; b < j->kw; ++b)
          acc += j->f[a * j->kw + b] * pd[(m + j->kh - 1 - a) * Wp + (l + j->kw - 1 - b)];
      fl[m * Wf + l] = acc;
    }
  /* 4. downsample: keep every down-th pixel */
  const int64_t Ho = oracle_upfirdn2d_out_len(j->H, j->up, j->down, j->py0, j->py1, j->kh);
  const int64_t Wo = oracle_upfirdn2d_out_len(j->W, j->up, j->down, j->px0, j->px1, j->kw);
  for (int64_t oh = 0; oh < Ho; ++oh)
    for (int64_t ow = 0; ow < Wo; ++ow)
      j->y[((n * Ho + oh) * Wo + ow) * j->C + c] = fl[(oh * j->down) * Wf + ow * j->down];
  free(u);
  free(pd);
  free(fl);
}

void oracle_upfirdn2d_f64(const double* x, const double* f, double* y, int64_t N, int64_t H,
                          int64_t W, int64_t C, int64_t up, int64_t down, int64_t px0, int64_t px1,
                          int64_t py0, int64_t py1, int64_t kh, int64_t kw) {
  ufd_job_t j = {x, f, y, N, H, W, C, up, down, px0, px1, py0, py1, kh, kw, NULL};
  ufd_parallel_for(N * C, ufd_plane, &j);
}

/* Sampled form for full-size checks: out[i] = y at linear NHWC index idx[i],
 * the four steps composed for that one output -- the downsampled position
 * (oh * down, ow * down) of the filtered plane reads padded positions
 * (oh * down + kh - 1 - a, ...), which hold the input pixel ((p - py0) / up)
 * when p - py0 is a non-negative multiple of up inside the upsampled plane
 * and zero otherwise. */
static void ufd_at_item(void* ctx, int64_t i) {
  const ufd_job_t* j = (const ufd_job_t*)ctx;
  const int64_t Ho = oracle_upfirdn2d_out_len(j->H, j->up, j->down, j->py0, j->py1, j->kh);
  const int64_t Wo = oracle_upfirdn2d_out_len(j->W, j->up, j->down, j->px0, j->px1, j->kw);
  const int64_t e = j->idx[i];
  const int64_t c = e % j->C, p = e / j->C;
  const int64_t ow = p % Wo, oh = (p / Wo) % Ho, n = p / (Wo * Ho);
  double acc = 0.0;
  for (int64_t a = 0; a < j->kh; ++a) {
    const int64_t ru = oh * j->down + j->kh - 1 - a - j->py0; /* row in the upsampled plane */
    if (ru < 0 || ru >= j->H * j->up || ru % j->up != 0) continue;
    for (int64_t b = 0; b < j->kw; ++b) {
      const int64_t cu = ow * j->down + j->kw - 1 - b - j->px0;
      if (cu < 0 || cu >= j->W * j->up || cu % j->up != 0) continue;
      acc += j->f[a * j->kw + b] * j->x[((n * j->H + ru / j->up) * j->W + cu / j->up) * j->C + c];
    }
  }
  j->y[i] = acc;
}

void oracle_upfirdn2d_at_f64(const double* x, const double* f, int64_t N, int64_t H, int64_t W,
                             int64_t C, int64_t up, int64_t down, int64_t px0, int64_t px1,
                             int64_t py0, int64_t py1, int64_t kh, int64_t kw, const int64_t* idx,
                             int64_t count, double* out) {
  ufd_job_t j = {x, f, out, N, H, W, C, up, down, px0, px1, py0, py1, kh, kw, idx};
  ufd_parallel_for(count, ufd_at_item, &j);
}
