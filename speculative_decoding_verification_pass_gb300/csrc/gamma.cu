// Dynamic speculation depth ("Build a Speculative Decoding Engine to Cut LLM
// Latency by 3x", Speculation Depth Tuning and Tree Drafting; Dynamic Gamma
// Controller).  Host code only: after each pass the caller records every
// slot's depth and accepted count (read back from spec_accept's n_accepted);
// each slot keeps a ring of its last `window` passes and, once `min_records`
// are in, takes the depth in [gamma_min, gamma_max] that maximises expected
// tokens per millisecond,
//   E(alpha, g) / (g * draft_ms_per_token + target_ms_per_pass),
//   E(alpha, g) = (1 - alpha^(g+1)) / (1 - alpha)   (g + 1 at alpha >= 1),
// alpha = accepted drafts / drafted tokens over the window (the prior while
// the window is empty).  Ties go to the smaller depth.
#include <cmath>
#include <new>
#include <vector>

#include "internal.h"

struct spec_gamma_ctl {
  int slots, gmin, gmax, ginit, window, min_records;
  double t_draft, t_target, prior;
  std::vector<int32_t> acc, drafted;  // [slots][window] ring of passes
  std::vector<int32_t> head, count, gamma;
  std::vector<int64_t> sum_acc, sum_drafted;
};

namespace {

double expected_tokens(double alpha, int g) {
  if (alpha >= 1.0) return static_cast<double>(g + 1);
  return (1.0 - std::pow(alpha, g + 1)) / (1.0 - alpha);
}

int best_gamma(double alpha, int gmin, int gmax, double t_draft, double t_target) {
  int best = gmin;
  double best_rate = -1.0;
  for (int g = gmin; g <= gmax; ++g) {
    const double rate = expected_tokens(alpha, g) / (g * t_draft + t_target);
    if (rate > best_rate) {
      best_rate = rate;
      best = g;
    }
  }
  return best;
}

double slot_alpha(const spec_gamma_ctl* c, int s) {
  return c->sum_drafted[s] > 0
             ? static_cast<double>(c->sum_acc[s]) / static_cast<double>(c->sum_drafted[s])
             : c->prior;
}

void slot_clear(spec_gamma_ctl* c, int s, int gamma_init) {
  c->head[s] = 0;
  c->count[s] = 0;
  c->sum_acc[s] = 0;
  c->sum_drafted[s] = 0;
  c->gamma[s] = gamma_init;
}

}  // namespace

extern "C" {

int spec_gamma_optimal(double alpha, int gamma_min, int gamma_max, double draft_ms_per_token,
                       double target_ms_per_pass, int32_t* out_gamma) {
  if (!out_gamma || !(alpha >= 0.0) || gamma_min < 0 || gamma_max < gamma_min) return SPEC_EINVAL;
  if (!(draft_ms_per_token >= 0.0) || !(target_ms_per_pass > 0.0)) return SPEC_EINVAL;
  *out_gamma = best_gamma(alpha > 1.0 ? 1.0 : alpha, gamma_min, gamma_max, draft_ms_per_token,
                          target_ms_per_pass);
  return SPEC_OK;
}

int spec_gamma_ctl_create(int slots, int gamma_min, int gamma_max, int gamma_init, int window,
                          int min_records, double draft_ms_per_token, double target_ms_per_pass,
                          double alpha_prior, spec_gamma_ctl** out) {
  if (!out) return SPEC_EINVAL;
  *out = nullptr;
  if (slots <= 0 || gamma_min < 0 || gamma_max < gamma_min || gamma_init < gamma_min ||
      gamma_init > gamma_max || window <= 0 || min_records < 0 || min_records > window)
    return SPEC_EINVAL;
  if (!(draft_ms_per_token >= 0.0) || !(target_ms_per_pass > 0.0)) return SPEC_EINVAL;
  if (!(alpha_prior >= 0.0 && alpha_prior <= 1.0)) return SPEC_EINVAL;
  if (static_cast<long long>(slots) * window > (1ll << 28)) return SPEC_ESIZE;
  spec_gamma_ctl* c = new (std::nothrow) spec_gamma_ctl();
  if (!c) return SPEC_ESIZE;
  c->slots = slots;
  c->gmin = gamma_min;
  c->gmax = gamma_max;
  c->ginit = gamma_init;
  c->window = window;
  c->min_records = min_records;
  c->t_draft = draft_ms_per_token;
  c->t_target = target_ms_per_pass;
  c->prior = alpha_prior;
  try {
    c->acc.assign(static_cast<size_t>(slots) * window, 0);
    c->drafted.assign(static_cast<size_t>(slots) * window, 0);
    c->head.assign(slots, 0);
    c->count.assign(slots, 0);
    c->gamma.assign(slots, gamma_init);
    c->sum_acc.assign(slots, 0);
    c->sum_drafted.assign(slots, 0);
  } catch (...) {
    delete c;
    return SPEC_ESIZE;
  }
  *out = c;
  return SPEC_OK;
}

int spec_gamma_ctl_destroy(spec_gamma_ctl* c) {
  delete c;
  return SPEC_OK;
}

int spec_gamma_ctl_reset(spec_gamma_ctl* c, int slot) {
  if (!c || slot < 0 || slot >= c->slots) return SPEC_EINVAL;
  slot_clear(c, slot, c->ginit);
  return SPEC_OK;
}

int spec_gamma_ctl_step(spec_gamma_ctl* c, int n, const int32_t* h_slot, const int32_t* h_gamma_used,
                        const int32_t* h_n_accepted, int32_t* h_gamma_next) {
  if (!c || n < 0 || (n > 0 && (!h_slot || !h_gamma_used || !h_n_accepted || !h_gamma_next)))
    return SPEC_EINVAL;
  // validate everything first: an invalid entry changes no slot
  for (int i = 0; i < n; ++i) {
    const int s = h_slot[i], g = h_gamma_used[i], a = h_n_accepted[i];
    if (s < 0 || s >= c->slots || g < 0 || a < 0 || a > g) return SPEC_EINVAL;
  }
  for (int i = 0; i < n; ++i) {
    const int s = h_slot[i];
    const size_t base = static_cast<size_t>(s) * c->window;
    if (c->count[s] == c->window) {  // the oldest pass leaves the window
      const size_t k = base + c->head[s];
      c->sum_acc[s] -= c->acc[k];
      c->sum_drafted[s] -= c->drafted[k];
    } else {
      ++c->count[s];
    }
    const size_t k = base + c->head[s];
    c->acc[k] = h_n_accepted[i];
    c->drafted[k] = h_gamma_used[i];
    c->sum_acc[s] += h_n_accepted[i];
    c->sum_drafted[s] += h_gamma_used[i];
    c->head[s] = (c->head[s] + 1) % c->window;
    if (c->count[s] >= c->min_records)
      c->gamma[s] = best_gamma(slot_alpha(c, s), c->gmin, c->gmax, c->t_draft, c->t_target);
    h_gamma_next[i] = c->gamma[s];
  }
  return SPEC_OK;
}

int spec_gamma_ctl_state(const spec_gamma_ctl* c, int slot, double* out_alpha, int32_t* out_gamma,
                         int32_t* out_records) {
  if (!c || slot < 0 || slot >= c->slots) return SPEC_EINVAL;
  if (out_alpha) *out_alpha = slot_alpha(c, slot);
  if (out_gamma) *out_gamma = c->gamma[slot];
  if (out_records) *out_records = c->count[slot];
  return SPEC_OK;
}

}  // extern "C"
