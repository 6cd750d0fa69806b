/*
 * CPU oracle for NHWC 2-D convolution: forward, weight gradient, bias
 * gradient and data gradient, written as the plain nested-loop definitions in
 * fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library. The product path never calls it and
 * shares no code, header, table or helper with it.
 *
 * What it follows:
 *  - The operation is the one PyTorch's nn.Conv2d performs (a cross-correlation
 *    over an NHWC input), whose weight.grad and bias.grad the page
 *    "ROCm/rocm-libraries PR #11188" ("Motivation") shows going to zero and
 *    staying correct, respectively. bias.grad is the sum of dY over every
 *    position; a 1x1 weight.grad equals the F.linear (GEMM) form on the
 *    reshaped tensors ("Motivation", "Test Plan").
 *  - Output extent: Ho = floor((H + 2 ph - dh (R - 1) - 1) / sh) + 1, the
 *    standard definition of a strided, dilated, zero-padded correlation (the
 *    pages do not print it).
 *  - Groups: output channel k reads input channels g*Cg .. g*Cg + Cg - 1 with
 *    g = floor(k / Kg), PyTorch's contiguous block mapping (the pages name
 *    grouped "cpg4/8" and depthwise problems in "perf(rocke): depthwise 7x7 and
 *    grouped cpg4/8 wgrad ..." ("Technical Details") but never print the
 *    mapping).
 *  - Split-K (the forward's or wgrad's reduction cut into slices that are
 *    summed afterwards, "feat(rocke): split-K forward implicit-GEMM convolution
 *    on gfx1250", "Two-stage split-K") changes only the order of the same sum,
 *    so the oracle has no split: it is the unsplit sum.
 *  - Batch split (PR #11188, "Technical Details"): the smallest number of
 *    dispatches m whose chunks hold at most max_n samples each, found by
 *    trying m = 1, 2, ... rather than by the page's closed form.
 *
 * Every product of two inputs is formed in double, where it is exact (two
 * 24-bit significands), and summed in double in the loop order written here:
 * wgrad sums over (n, ho, wo) in increasing order, forward over (r, s, c),
 * dgrad over (r, s, k).
 * Threads split the OUTPUTS among themselves; no output's sum is reordered.
 * Build with -ffp-contract=off so no multiply-add is fused.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int64_t n, h, w, c, k, r, s;
  int64_t stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, groups;
} oracle_problem;

/* Ho (or Wo): floor((in + 2 pad - dil (f - 1) - 1) / stride) + 1, or 0 when
 * the dilated filter does not fit in the padded input. */
int64_t oracle_out_extent(int64_t in, int64_t pad, int64_t dil, int64_t f, int64_t stride) {
  int64_t span = in + 2 * pad - dil * (f - 1) - 1;
  if (span < 0 || stride < 1) return 0;
  return span / stride + 1;
}

/* ---------------------------------------------------------------- threads */

typedef struct {
  const oracle_problem* p;
  const float* x;
  const float* wt; /* weight (fwd) */
  const float* dy; /* output gradient (wgrad) */
  double* out;
  int64_t lo, hi; /* the outputs this worker owns (meaning depends on the op) */
} work;

/* Runs fn on nthreads workers; worker t owns [first + total*t/nt, first + total*(t+1)/nt). */
static void run_parallel(void* (*fn)(void*), const work* base, int64_t first, int64_t total,
                         int nthreads) {
  if (total <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > total) nthreads = (int)(total > 0 ? total : 1);
  work* jobs = (work*)malloc(sizeof(work) * (size_t)nthreads);
  pthread_t* tids = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  int* ok = (int*)calloc((size_t)nthreads, sizeof(int));
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *base;
    jobs[t].lo = first + total * t / nthreads;
    jobs[t].hi = first + total * (t + 1) / nthreads;
    if (t > 0) ok[t] = pthread_create(&tids[t], NULL, fn, &jobs[t]) == 0;
  }
  fn(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (ok[t]) pthread_join(tids[t], NULL);
    else fn(&jobs[t]);
  }
  free(ok);
  free(tids);
  free(jobs);
}

/* ---------------------------------------------------------------- forward */

/* Y[n,ho,wo,k] = sum over r, s, c < Cg of
 *   X[n, ho*sh + r*dh - ph, wo*sw + s*dw - pw, g*Cg + c] * W[k, r, s, c],
 * terms with the input position outside [0,H) x [0,W) being zero.
 * This worker owns output rows (n, ho) in [lo, hi). */
static void* fwd_worker(void* arg) {
  const work* j = (const work*)arg;
  const oracle_problem* p = j->p;
  const int64_t Ho = oracle_out_extent(p->h, p->pad_h, p->dil_h, p->r, p->stride_h);
  const int64_t Wo = oracle_out_extent(p->w, p->pad_w, p->dil_w, p->s, p->stride_w);
  const int64_t Cg = p->c / p->groups, Kg = p->k / p->groups;
  for (int64_t row = j->lo; row < j->hi; ++row) {
    const int64_t n = row / Ho, ho = row % Ho;
    for (int64_t wo = 0; wo < Wo; ++wo) {
      for (int64_t k = 0; k < p->k; ++k) {
        const int64_t g = k / Kg;
        double acc = 0.0;
        for (int64_t r = 0; r < p->r; ++r) {
          const int64_t h = ho * p->stride_h + r * p->dil_h - p->pad_h;
          if (h < 0 || h >= p->h) continue;
          for (int64_t s = 0; s < p->s; ++s) {
            const int64_t w = wo * p->stride_w + s * p->dil_w - p->pad_w;
            if (w < 0 || w >= p->w) continue;
            const float* xp = j->x + ((n * p->h + h) * p->w + w) * p->c + g * Cg;
            const float* wp = j->wt + ((k * p->r + r) * p->s + s) * Cg;
            for (int64_t c = 0; c < Cg; ++c) acc += (double)xp[c] * (double)wp[c];
          }
        }
        j->out[((n * Ho + ho) * Wo + wo) * p->k + k] = acc;
      }
    }
  }
  return NULL;
}

void oracle_conv_fwd(const oracle_problem* p, const float* x, const float* wt, double* y,
                     int nthreads) {
  const int64_t Ho = oracle_out_extent(p->h, p->pad_h, p->dil_h, p->r, p->stride_h);
  work base = {p, x, wt, NULL, y, 0, 0};
  run_parallel(fwd_worker, &base, 0, p->n * Ho, nthreads);
}

/* ------------------------------------------------------------ weight grad */

/* dW[k,r,s,c] += sum over (n, ho, wo) of
 *   dY[n,ho,wo,k] * X[n, ho*sh + r*dh - ph, wo*sw + s*dw - pw, g*Cg + c].
 * This worker owns output channels k in [lo, hi). */
static void* wgrad_worker(void* arg) {
  const work* j = (const work*)arg;
  const oracle_problem* p = j->p;
  const int64_t Ho = oracle_out_extent(p->h, p->pad_h, p->dil_h, p->r, p->stride_h);
  const int64_t Wo = oracle_out_extent(p->w, p->pad_w, p->dil_w, p->s, p->stride_w);
  const int64_t Cg = p->c / p->groups, Kg = p->k / p->groups;
  for (int64_t n = 0; n < p->n; ++n) {
    for (int64_t ho = 0; ho < Ho; ++ho) {
      for (int64_t wo = 0; wo < Wo; ++wo) {
        const float* dyp = j->dy + ((n * Ho + ho) * Wo + wo) * p->k;
        for (int64_t k = j->lo; k < j->hi; ++k) {
          const double gk = (double)dyp[k];
          const int64_t g = k / Kg;
          for (int64_t r = 0; r < p->r; ++r) {
            const int64_t h = ho * p->stride_h + r * p->dil_h - p->pad_h;
            if (h < 0 || h >= p->h) continue;
            for (int64_t s = 0; s < p->s; ++s) {
              const int64_t w = wo * p->stride_w + s * p->dil_w - p->pad_w;
              if (w < 0 || w >= p->w) continue;
              const float* xp = j->x + ((n * p->h + h) * p->w + w) * p->c + g * Cg;
              double* d = j->out + ((k * p->r + r) * p->s + s) * Cg;
              for (int64_t c = 0; c < Cg; ++c) d[c] += gk * (double)xp[c];
            }
          }
        }
      }
    }
  }
  return NULL;
}

/* Adds the contribution of all p->n samples in x / dy to dw for output
 * channels [k_begin, k_end). dw is the full [K][R][S][Cg] array. Calling it
 * on consecutive batch chunks adds the same terms in the same order as one
 * call on the whole batch. */
void oracle_conv_wgrad_acc(const oracle_problem* p, const float* x, const float* dy,
                           int64_t k_begin, int64_t k_end, double* dw, int nthreads) {
  if (k_begin < 0) k_begin = 0;
  if (k_end > p->k) k_end = p->k;
  if (k_end <= k_begin) return;
  work base = {p, x, NULL, dy, dw, 0, 0};
  run_parallel(wgrad_worker, &base, k_begin, k_end - k_begin, nthreads);
}

/* -------------------------------------------------------------- data grad */

/* dX[n,h,w,g*Cg + c] = sum over k = g*Kg .. g*Kg + Kg - 1, r, s of
 *   dY[n,ho,wo,k] * W[k,r,s,c]
 * for the one (ho, wo) per tap with ho*sh + r*dh - ph = h and
 * wo*sw + s*dw - pw = w inside [0,Ho) x [0,Wo): the forward output positions
 * that read input (h, w) through tap (r, s). This is the gradient of the
 * forward with respect to X (the "dgrad" direction the split-K resolver of
 * "feat(rocke): split-K forward implicit-GEMM convolution on gfx1250",
 * "Auto-deduced degree", also covers). Summed over r, then s, then k.
 * This worker owns input rows (n, h) in [lo, hi). */
static void* dgrad_worker(void* arg) {
  const work* j = (const work*)arg;
  const oracle_problem* p = j->p;
  const int64_t Ho = oracle_out_extent(p->h, p->pad_h, p->dil_h, p->r, p->stride_h);
  const int64_t Wo = oracle_out_extent(p->w, p->pad_w, p->dil_w, p->s, p->stride_w);
  const int64_t Cg = p->c / p->groups, Kg = p->k / p->groups;
  for (int64_t row = j->lo; row < j->hi; ++row) {
    const int64_t n = row / p->h, h = row % p->h;
    for (int64_t w = 0; w < p->w; ++w) {
      for (int64_t ci = 0; ci < p->c; ++ci) {
        const int64_t g = ci / Cg, c = ci % Cg;
        double acc = 0.0;
        for (int64_t r = 0; r < p->r; ++r) {
          const int64_t hn = h + p->pad_h - r * p->dil_h; /* = ho * sh */
          if (hn < 0 || hn % p->stride_h != 0) continue;
          const int64_t ho = hn / p->stride_h;
          if (ho >= Ho) continue;
          for (int64_t s = 0; s < p->s; ++s) {
            const int64_t wn = w + p->pad_w - s * p->dil_w; /* = wo * sw */
            if (wn < 0 || wn % p->stride_w != 0) continue;
            const int64_t wo = wn / p->stride_w;
            if (wo >= Wo) continue;
            const float* dyp = j->dy + ((n * Ho + ho) * Wo + wo) * p->k + g * Kg;
            const float* wp = j->wt + ((g * Kg * p->r + r) * p->s + s) * Cg + c;
            for (int64_t kk = 0; kk < Kg; ++kk)
              acc += (double)dyp[kk] * (double)wp[kk * p->r * p->s * Cg];
          }
        }
        j->out[((n * p->h + h) * p->w + w) * p->c + ci] = acc;
      }
    }
  }
  return NULL;
}

void oracle_conv_dgrad(const oracle_problem* p, const float* dy, const float* wt, double* dx,
                       int nthreads) {
  work base = {p, NULL, wt, dy, dx, 0, 0};
  run_parallel(dgrad_worker, &base, 0, p->n * p->h, nthreads);
}

/* -------------------------------------------------------------- bias grad */

/* db[k] += sum over (n, ho, wo) of dY[n,ho,wo,k] (PR #11188, "Motivation":
 * bias.grad, the gradient that stayed correct). */
void oracle_conv_bgrad_acc(const oracle_problem* p, const float* dy, double* db) {
  const int64_t Ho = oracle_out_extent(p->h, p->pad_h, p->dil_h, p->r, p->stride_h);
  const int64_t Wo = oracle_out_extent(p->w, p->pad_w, p->dil_w, p->s, p->stride_w);
  const int64_t P = p->n * Ho * Wo;
  for (int64_t q = 0; q < P; ++q)
    for (int64_t k = 0; k < p->k; ++k) db[k] += (double)dy[q * p->k + k];
}

/* ------------------------------------------------------------ batch split */

/* The smallest number of dispatches m such that m chunks of at most max_n
 * samples can hold all n samples (PR #11188, "Motivation": no dispatch may
 * address more than the limit). Found by trying m = 1, 2, ...; returns -1 for
 * max_n < 1 or n < 0. */
int64_t oracle_batch_split_count(int64_t n, int64_t max_n) {
  if (max_n < 1 || n < 0) return -1;
  int64_t m = 1;
  while (m * max_n < n) ++m;
  return m;
}
