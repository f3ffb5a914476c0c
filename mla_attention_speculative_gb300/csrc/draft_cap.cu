// Draft-cap selection from a measured verify-cost curve (mla_select_draft_cap).
//
// "Draft caps and calibration" (mlx-dspark docs): a cap C is how many drafted
// tokens are verified per round, and the engine derives the best fixed cap
// from its measured curves with the cost model it gives "in formula form":
//   speedup(C) = accepted(C) / (drafter + verify(C + 1)),
//   accepted(C) = 1 + p + ... + p^C   (tokens committed per round),
//   verify(w)  = the cost of one verify pass over w rows, in single-token steps.
// Costs arrive in any unit and are expressed in single-token steps by
// dividing by verify(1); C = 0 is plain decoding (speedup 1, no drafter);
// the drafter's cost is one number for all caps or one per cap; ties go to
// the smaller cap.  Host code only: the verify curve is what the library's
// own kernels measure (µs per call against L).

#include <cmath>

#include "mla_internal.h"

namespace {

// 1 + p + ... + p^C, summed term by term.
double accepted_tokens(double p, int C) {
  double total = 0.0, term = 1.0;
  for (int i = 0; i <= C; ++i) {
    total += term;
    term *= p;
  }
  return total;
}

}  // namespace

extern "C" int32_t mla_select_draft_cap(double p, const double* verify_cost, int32_t n_verify,
                                        const double* drafter_cost, int32_t n_drafter,
                                        int32_t max_cap, double* speedup_out) {
  using mla::set_error;
  if (!(p >= 0.0 && p <= 1.0)) {
    set_error("acceptance probability %g is outside [0, 1]", p);
    return -1;
  }
  if (verify_cost == nullptr || n_verify < 1 || drafter_cost == nullptr || n_drafter < 1 ||
      max_cap < 0) {
    set_error("draft cap needs a verify curve, a drafter cost and max_cap >= 0");
    return -1;
  }
  for (int32_t i = 0; i < n_verify; ++i) {
    if (!(verify_cost[i] > 0.0) || !std::isfinite(verify_cost[i])) {
      set_error("verify_cost[%d] = %g is not a positive cost", i, verify_cost[i]);
      return -1;
    }
  }
  for (int32_t i = 0; i < n_drafter; ++i) {
    if (!(drafter_cost[i] >= 0.0) || !std::isfinite(drafter_cost[i])) {
      set_error("drafter_cost[%d] = %g is not a cost", i, drafter_cost[i]);
      return -1;
    }
  }
  int32_t limit = max_cap < n_verify - 1 ? max_cap : n_verify - 1;
  if (n_drafter > 1 && limit > n_drafter - 1) limit = n_drafter - 1;
  const double step = verify_cost[0];  // one plain decode step
  int32_t best = 0;
  double best_s = 1.0;
  if (speedup_out) speedup_out[0] = 1.0;
  for (int32_t C = 1; C <= limit; ++C) {
    const double d = n_drafter == 1 ? drafter_cost[0] : drafter_cost[C];
    const double s = accepted_tokens(p, C) * step / (d + verify_cost[C]);
    if (speedup_out) speedup_out[C] = s;
    if (s > best_s) {
      best_s = s;
      best = C;
    }
  }
  return best;
}
