// Host-side analysis of speculative decoding rounds, for choosing the draft
// length k online ("投机解码:为什么一个字都不改", the bookkeeping section and
// its three experiments; the pages defer the choice of k under a draft cost
// to Leviathan et al., appendix A.1 and theorem 3.8):
//   - expected tokens per round when each of the k positions is accepted
//     independently with probability alpha: (1 - alpha^(k+1)) / (1 - alpha);
//   - walltime speedup when one draft forward costs c target forwards: a
//     round costs k c + 1 forwards, so speedup = tokens per round / (k c + 1);
//   - the k in [0, k_max] with the largest speedup (k = 0 is plain decoding,
//     speedup 1);
//   - alpha estimated from observed rounds: a round with draft length L that
//     accepted m tested m + 1 positions when m < L and m when m = L, of which
//     m were accepted, so the estimate is sum(m) / sum(tests) (the maximum
//     likelihood estimate for independent Bernoulli(alpha) positions).
// Plain host code: no GPU, no CUDA calls.
#include <cmath>

#include "spec_verify.h"

namespace {

double tokens_per_round(double alpha, int k) {
  if (alpha >= 1.0) return k + 1.0;
  // 1 + alpha + ... + alpha^k, summed directly: exact for alpha = 0 and
  // without the cancellation of 1 - alpha^(k+1) near alpha = 1
  double sum = 0.0, term = 1.0;
  for (int i = 0; i <= k; ++i) {
    sum += term;
    term *= alpha;
  }
  return sum;
}

bool valid_alpha(double alpha) { return alpha >= 0.0 && alpha <= 1.0; }

}  // namespace

extern "C" {

int spec_expected_tokens(double alpha, int k, double *out) {
  if (!out || !valid_alpha(alpha) || k < 0) return SPEC_EINVAL;
  *out = tokens_per_round(alpha, k);
  return SPEC_OK;
}

int spec_speedup(double alpha, int k, double draft_cost, double *out) {
  if (!out || !valid_alpha(alpha) || k < 0 || !(draft_cost >= 0.0) || !std::isfinite(draft_cost))
    return SPEC_EINVAL;
  *out = tokens_per_round(alpha, k) / (k * draft_cost + 1.0);
  return SPEC_OK;
}

int spec_best_k(double alpha, double draft_cost, int k_max, int *k_out, double *speedup_out) {
  if (!k_out || !valid_alpha(alpha) || k_max < 0 || !(draft_cost >= 0.0) || !std::isfinite(draft_cost))
    return SPEC_EINVAL;
  int best = 0;
  double best_s = 1.0;
  for (int k = 1; k <= k_max; ++k) {
    const double s = tokens_per_round(alpha, k) / (k * draft_cost + 1.0);
    if (s > best_s) {  // ties keep the shorter draft
      best = k;
      best_s = s;
    }
  }
  *k_out = best;
  if (speedup_out) *speedup_out = best_s;
  return SPEC_OK;
}

int spec_alpha_estimate(const int32_t *accepted, const int32_t *draft_len, int n, int k, double *alpha_out,
                        int64_t *tests_out) {
  if (!alpha_out || n < 0 || (n > 0 && !accepted) || k < 0) return SPEC_EINVAL;
  long long acc = 0, tests = 0;
  for (int r = 0; r < n; ++r) {
    const int L = draft_len ? draft_len[r] : k;
    const int m = accepted[r];
    if (L < 0 || m < 0 || m > L) return SPEC_EINVAL;
    acc += m;
    tests += m + (m < L ? 1 : 0);
  }
  *alpha_out = tests > 0 ? static_cast<double>(acc) / static_cast<double>(tests) : NAN;
  if (tests_out) *tests_out = tests;
  return SPEC_OK;
}

}  // extern "C"
