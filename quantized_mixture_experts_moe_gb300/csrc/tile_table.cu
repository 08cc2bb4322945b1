// The tile table: per-shape choices of the token tile (NMAX), set by the
// caller from a measured sweep, in the manner of the tuned grouped-fmoe
// configuration rows (the aiter tuned grouped-fmoe page, Changes: one row per
// model shape, TP degree and token bucket).  The rules are host state read at
// launch time by every call that sizes or schedules token tiles.
#include "mx_tiles.cuh"
#include "qmoe_common.cuh"

#include <mutex>
#include <vector>

namespace qmoe {
namespace {

std::mutex g_mu;
std::vector<qmoe_tile_rule> g_rules;

bool matches(const qmoe_tile_rule& r, const qmoe_dims* d) {
    const int64_t T = d->T;
    return (r.H == 0 || r.H == d->H) && (r.I == 0 || r.I == d->I) && (r.E == 0 || r.E == d->E) &&
           (r.k == 0 || r.k == d->k) && T >= r.t_min && T <= r.t_max;
}

}  // namespace

namespace mxt {
int nmax_for(const qmoe_dims* d) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (const qmoe_tile_rule& r : g_rules)
        if (matches(r, d)) return r.nmax;
    return nmax_default(d);
}
}  // namespace mxt

}  // namespace qmoe

extern "C" int qmoe_set_tile_rules(const qmoe_tile_rule* rules, int n) {
    if (n < 0 || (n > 0 && !rules) || n > 4096) return QMOE_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        const qmoe_tile_rule& r = rules[i];
        if ((r.nmax != 16 && r.nmax != 112 && r.nmax != 224) || r.H < 0 || r.I < 0 || r.E < 0 || r.k < 0 || r.t_min < 0 ||
            r.t_max < r.t_min)
            return QMOE_ERR_ARG;
    }
    std::lock_guard<std::mutex> lock(qmoe::g_mu);
    qmoe::g_rules.assign(rules, rules + n);
    return QMOE_OK;
}

extern "C" int qmoe_tile_nmax(const qmoe_dims* d) {
    if (!d) return QMOE_ERR_ARG;
    return qmoe::mxt::nmax_for(d);
}
