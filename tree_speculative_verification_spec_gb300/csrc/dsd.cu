// Dynamic draft length ("Hardware-aware dynamic speculative decoding"):
// the offline goodput table (goodput = AL / ITL), its runtime lookup, live
// statistics folded into it, and the <tokens, K> keys of the full CUDA graphs
// to capture.  Host code: the scheduler runs it between steps.
#include <cmath>

#include "common.cuh"

extern "C" {

spec_status spec_dsd_optimal_k(const double* al, const double* itl, int n_bs, int n_k, const int32_t* k_values,
                               int32_t* k_opt) {
  if (n_bs < 0 || n_k < 0) return SPEC_ERR_INVALID_ARG;
  if (n_bs == 0) return SPEC_OK;
  if (!k_opt || (n_k > 0 && (!al || !itl || !k_values))) return SPEC_ERR_INVALID_ARG;
  for (int b = 0; b < n_bs; ++b) {
    const double* a = al + (size_t)b * n_k;
    const double* t = itl + (size_t)b * n_k;
    int arg = -1;
    double g_best = 0.0;
    for (int j = 0; j < n_k; ++j) {
      if (!std::isfinite(a[j]) || !std::isfinite(t[j]) || t[j] <= 0.0) continue;  // unmeasured cell
      const double g = a[j] / t[j];
      if (arg < 0 || g > g_best) {  // strict: the earliest column keeps a tie
        arg = j;
        g_best = g;
      }
    }
    k_opt[b] = arg >= 0 ? k_values[arg] : -1;
  }
  return SPEC_OK;
}

spec_status spec_dsd_select_k(const int32_t* bs_table, const int32_t* k_table, int n, int bs, int32_t* k_out) {
  if (n <= 0 || !bs_table || !k_table || !k_out) return SPEC_ERR_INVALID_ARG;
  for (int i = 1; i < n; ++i)
    if (bs_table[i] <= bs_table[i - 1]) return SPEC_ERR_INVALID_ARG;  // must ascend strictly
  // binary search for the last entry with bs_table[i] <= bs
  int lo = 0, hi = n;  // answer in [lo, hi)
  if (bs < bs_table[0]) {
    *k_out = k_table[0];
    return SPEC_OK;
  }
  while (hi - lo > 1) {
    const int mid = lo + (hi - lo) / 2;
    if (bs_table[mid] <= bs) lo = mid;
    else hi = mid;
  }
  *k_out = k_table[lo];
  return SPEC_OK;
}

spec_status spec_dsd_update(double* al, double* itl, int n_bs, int n_k, int bs_index, int k_index, double al_sample,
                            double itl_sample, double weight) {
  if (!al || !itl || n_bs <= 0 || n_k <= 0 || bs_index < 0 || bs_index >= n_bs || k_index < 0 || k_index >= n_k)
    return SPEC_ERR_INVALID_ARG;
  if (!(weight > 0.0 && weight <= 1.0) || !std::isfinite(al_sample) || !std::isfinite(itl_sample))
    return SPEC_ERR_INVALID_ARG;
  const size_t c = (size_t)bs_index * n_k + k_index;
  al[c] = std::isfinite(al[c]) ? al[c] + weight * (al_sample - al[c]) : al_sample;
  itl[c] = std::isfinite(itl[c]) ? itl[c] + weight * (itl_sample - itl[c]) : itl_sample;
  return SPEC_OK;
}

spec_status spec_dsd_graph_keys(int max_tokens, int max_k, int32_t* tokens_out, int32_t* k_out, int cap,
                                int32_t* count) {
  if (max_tokens < 0 || max_k < 0 || cap < 0 || !count || (cap > 0 && (!tokens_out || !k_out)))
    return SPEC_ERR_INVALID_ARG;
  long long n = 0;
  for (int t = 2; t <= max_tokens; ++t) {
    // K + 1 ranges over the divisors d of t with 2 <= d <= max_k + 1
    const int dmax = max_k + 1 < t ? max_k + 1 : t;
    for (int d = 2; d <= dmax; ++d) {
      if (t % d) continue;
      if (n < cap) {
        tokens_out[n] = t;
        k_out[n] = d - 1;
      }
      ++n;
    }
  }
  if (n > 0x7fffffff) return SPEC_ERR_UNSUPPORTED;
  *count = (int32_t)n;
  return SPEC_OK;
}

}  // extern "C"
