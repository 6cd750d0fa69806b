// Host sanitizer harness for the library's planner (built with -fsanitize=address,undefined by
// tests/test_sanitizers.py, with the kernels compiled in but never launched): validation, output
// extents, the split-K degree policy, workspace arithmetic and plan description over a grid of
// problems, directions, dtypes and degree requests, valid and invalid (negative, zero, NULL, and
// sizes at the int64 overflow edge). Any out-of-bounds access, signed overflow or other undefined
// behaviour in the host code stops the run.
#include <cstdint>
#include <cstdio>

#include "conv_igemm.h"

int main() {
  long long ok = 0, rejected = 0;
  const int64_t sizes[] = {1, 3, 7, 14, 28, 56};
  const int64_t chans[] = {1, 8, 32, 64, 96, 128, 256, 384, 512};
  const int64_t filters[] = {1, 2, 3, 5, 7};
  const int64_t groupsv[] = {1, 2, 4, 8, 64, 128, 384};
  const int32_t requests[] = {-2, -1, 0, 1, 2, 7, 33, 1000000};
  const int32_t sms[] = {1, 148, 152};
  for (int64_t hw : sizes)
    for (int64_t c : chans)
      for (int64_t f : filters)
        for (int64_t g : groupsv) {
          if (c % g != 0) continue;
          for (int dt = 0; dt < 3; ++dt)
            for (int st = 1; st <= 2; ++st) {
              conv_problem p{};
              p.n = hw == 1 ? 0 : 2;
              p.h = hw;
              p.w = hw + 1;
              p.c = c;
              p.k = c;
              p.r = f;
              p.s = f;
              p.stride_h = st;
              p.stride_w = st;
              p.pad_h = f / 2;
              p.pad_w = f / 2;
              p.dil_h = 1;
              p.dil_w = st;
              p.groups = g;
              p.in_dtype = dt;
              p.out_dtype = dt == 0 ? 0 : (st == 1 ? dt : 0);
              int64_t ho = 0, wo = 0;
              if (conv_output_dims(&p, &ho, &wo) != CONV_OK) {
                ++rejected;
                continue;
              }
              for (int dir = 0; dir < 3; ++dir)
                for (int32_t req : requests)
                  for (int32_t sm : sms) {
                    int32_t degree = 0;
                    uint64_t bytes = 0;
                    conv_plan_info info{};
                    const conv_status a = resolve_split_k_for(&p, (conv_dir)dir, req, sm, &degree);
                    const conv_status b = conv_workspace_bytes_for(&p, (conv_dir)dir, req, 1, sm, &bytes);
                    const conv_status c2 = conv_describe_plan(&p, (conv_dir)dir, req, 1, sm, &info);
                    if (a == CONV_OK && b == CONV_OK && c2 == CONV_OK) ++ok;
                    else ++rejected;
                  }
            }
        }
  // invalid problems and pointers
  conv_problem bad{};
  int64_t ho, wo;
  int32_t degree;
  uint64_t bytes;
  conv_plan_info info;
  rejected += conv_output_dims(nullptr, &ho, &wo) != CONV_OK;
  rejected += conv_output_dims(&bad, &ho, &wo) != CONV_OK;
  bad = conv_problem{1, 1, 1, 1, 1, 1, 1, 1, 1, 0, 0, 1, 1, 1, 0, 0};
  rejected += conv_output_dims(&bad, nullptr, &wo) != CONV_OK;
  rejected += resolve_split_k_for(&bad, CONV_DIR_FWD, -1, 152, nullptr) != CONV_OK;
  rejected += conv_workspace_bytes_for(&bad, (conv_dir)7, -1, 0, 152, &bytes) != CONV_OK;
  rejected += conv_describe_plan(&bad, CONV_DIR_WGRAD, -1, 0, 0, &info) != CONV_OK;
  // sizes at the overflow edge: every byte count must be checked, none may wrap
  const int64_t big = (int64_t)1 << 61;
  conv_problem huge{big, 2, 2, 2, 2, 1, 1, 1, 1, 0, 0, 1, 1, 1, 0, 0};
  rejected += conv_output_dims(&huge, &ho, &wo) != CONV_OK;
  rejected += conv_describe_plan(&huge, CONV_DIR_WGRAD, -1, 1, 152, &info) != CONV_OK;
  huge = conv_problem{1, 1, 1, 1, 1, 1, 1, 1, 1, INT64_MAX / 2, 0, INT64_MAX / 2, 1, 1, 0, 0};
  rejected += conv_output_dims(&huge, &ho, &wo) != CONV_OK;
  rejected += resolve_split_k_for(&huge, CONV_DIR_FWD, -1, 152, &degree) != CONV_OK;
  for (int64_t n = -3; n < 200; n += 5)
    for (int64_t m = -2; m < 60; m += 7) ok += conv_batch_split_count(n, m) > 0;
  ok += conv_batch_split_count(INT64_MAX, 1) > 0;
  std::printf("planner harness ok %lld plans, %lld rejected\n", ok, rejected);
  return 0;
}
