/* Host sanitizer harness for the CPU oracle (built with -fsanitize=address,undefined by
 * tests/test_sanitizers.py): runs every oracle entry point on small problems with strides,
 * dilations, padding and groups, plus its extent and batch-split helpers, so an out-of-bounds
 * access or undefined behaviour in the oracle's loops stops the run. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

typedef struct {
  int64_t n, h, w, c, k, r, s;
  int64_t stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, groups;
} oracle_problem;

int64_t oracle_out_extent(int64_t in, int64_t pad, int64_t dil, int64_t f, int64_t stride);
void oracle_conv_fwd(const oracle_problem* p, const float* x, const float* w, double* y, int nthreads);
void oracle_conv_wgrad_acc(const oracle_problem* p, const float* x, const float* dy, int64_t k_begin,
                           int64_t k_end, double* dw, int nthreads);
void oracle_conv_dgrad(const oracle_problem* p, const float* dy, const float* w, double* dx, int nthreads);
void oracle_conv_bgrad_acc(const oracle_problem* p, const float* dy, double* db);
int64_t oracle_batch_split_count(int64_t n, int64_t max_n);

static float* filled(int64_t n) {
  float* a = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  for (int64_t i = 0; i < n; ++i) a[i] = (float)((i * 2654435761u) % 17) - 8.0f;
  return a;
}

int main(void) {
  const oracle_problem probs[] = {
      {2, 7, 9, 6, 4, 3, 2, 1, 2, 1, 0, 1, 1, 2},
      {1, 8, 8, 8, 6, 3, 3, 2, 2, 1, 1, 2, 1, 2},
      {3, 5, 6, 4, 4, 5, 3, 1, 1, 2, 3, 1, 2, 4},
      {2, 9, 7, 12, 8, 1, 4, 3, 1, 0, 2, 1, 1, 4},
      {1, 4, 5, 8, 8, 3, 3, 1, 1, 0, 0, 1, 1, 8},
      {0, 4, 4, 4, 4, 3, 3, 1, 1, 1, 1, 1, 1, 1},
  };
  const int np = (int)(sizeof(probs) / sizeof(probs[0]));
  for (int i = 0; i < np; ++i) {
    const oracle_problem* p = &probs[i];
    const int64_t ho = oracle_out_extent(p->h, p->pad_h, p->dil_h, p->r, p->stride_h);
    const int64_t wo = oracle_out_extent(p->w, p->pad_w, p->dil_w, p->s, p->stride_w);
    const int64_t cg = p->c / p->groups;
    const int64_t nx = p->n * p->h * p->w * p->c, nw = p->k * p->r * p->s * cg, ny = p->n * ho * wo * p->k;
    float *x = filled(nx), *w = filled(nw), *dy = filled(ny);
    double* y = (double*)calloc((size_t)(ny > 0 ? ny : 1), sizeof(double));
    double* dw = (double*)calloc((size_t)nw, sizeof(double));
    double* dx = (double*)calloc((size_t)(nx > 0 ? nx : 1), sizeof(double));
    double* db = (double*)calloc((size_t)p->k, sizeof(double));
    for (int threads = 1; threads <= 3; threads += 2) {
      oracle_conv_fwd(p, x, w, y, threads);
      oracle_conv_wgrad_acc(p, x, dy, 0, p->k, dw, threads);
      oracle_conv_wgrad_acc(p, x, dy, 1, p->k - 1, dw, threads);
      oracle_conv_dgrad(p, dy, w, dx, threads);
    }
    oracle_conv_bgrad_acc(p, dy, db);
    free(x); free(w); free(dy); free(y); free(dw); free(dx); free(db);
  }
  int64_t acc = 0;
  for (int64_t n = -1; n < 300; n += 7)
    for (int64_t m = -1; m < 50; m += 3) acc += oracle_batch_split_count(n, m);
  acc += oracle_out_extent(5, 0, 3, 3, 1) + oracle_out_extent(1, 0, 1, 4, 1);
  printf("oracle harness ok %lld\n", (long long)acc);
  return 0;
}
