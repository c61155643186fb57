// kstar.cpp -- choice of the controller's reuse interval K* (EvoCG, "Self-Evolving Precision
// Control for Faster Conjugate Gradient", §3.4 interval reuse scheduling), on the host.
//
// From a run that decides every iteration, the log holds each column block's precision code
// per iteration (0 = FP64, 1 = FP32, 2 = BF16; a lower code is a higher precision). Reusing
// every K-th decision puts the decision of iteration K*floor(k/K) in force at iteration k.
// An upward transition (a block's code drops from iteration k-1 to k) is delayed under K
// when the decision in force at k has a higher code than iteration k's own. K* is the largest
// of 1, 2, 4, ... whose fraction of delayed upward transitions stays below the limit.
#include <cstdint>
#include <vector>

#include "evocg_internal.h"

extern "C" int evocg_kstar_select(const uint8_t *map_log, int64_t rows, int64_t ncb, double limit,
                                  int *kstar, double *fractions, int max_candidates, int *ncand)
{
    evocg::set_error("");
    if (rows < 0 || ncb < 1) return evocg::fail(EVOCG_EINVAL, "rows must be >= 0 and ncb >= 1");
    if (!kstar || (rows > 0 && !map_log)) return evocg::fail(EVOCG_EINVAL, "NULL argument");
    if (fractions && max_candidates < 0) return evocg::fail(EVOCG_EINVAL, "max_candidates < 0");
    for (int64_t i = 0; i < rows * ncb; ++i)
        if (map_log[i] > 2) return evocg::fail(EVOCG_EINVAL, "precision code above 2 in the log");

    // upward transitions once, as (iteration, block) pairs
    std::vector<int64_t> up_k, up_i;
    for (int64_t k = 1; k < rows; ++k) {
        const uint8_t *cur = map_log + k * ncb, *prev = cur - ncb;
        for (int64_t i = 0; i < ncb; ++i)
            if (cur[i] < prev[i]) {
                up_k.push_back(k);
                up_i.push_back(i);
            }
    }
    int best = 1, count = 0;
    for (int64_t K = 1; K <= (rows > 0 ? rows : 1); K *= 2) {
        int64_t delayed = 0;
        for (size_t u = 0; u < up_k.size(); ++u) {
            const int64_t k = up_k[u], i = up_i[u];
            const int64_t kr = (k / K) * K;   // the iteration whose decision is in force
            if (map_log[kr * ncb + i] > map_log[k * ncb + i]) ++delayed;
        }
        const double frac = up_k.empty() ? 0.0 : (double)delayed / (double)up_k.size();
        if (fractions && count < max_candidates) fractions[count] = frac;
        ++count;
        if (frac < limit && K > best) best = (int)K;
        if (K > (int64_t)1 << 29) break;
    }
    *kstar = best;
    if (ncand) *ncand = count;
    return EVOCG_OK;
}
