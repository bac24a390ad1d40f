// The polymerizer: per-shape choice of regions, micro-kernels and split-K
// factors under the cost model of the MikPoly summary, section 3
// ("polymerization cost model", "heuristic search").
//
//   Cost(S, H) = sum over regions (R_i, K~_i) of  f_wave * f_pipe  (+ tail)
//   f_wave     = ceil(f_parallel(R_i, K~_i) / |P_multi|)
//   f_pipe     = g_predict(f_num(R_i, K~_i))
//
// The tail is the section's three-stage pipeline taken at its word: a PE runs
// its tasks back to back, each task's write-back (stage 3) overlapping the
// next task's load and compute, so only the last wave's write-back is not
// hidden.  It is charged once per strategy (the largest tail among its
// regions' micro-kernels, with the launch and the pipeline fill), and
// g_predict keeps only what every task pays.
//
// f_parallel is the number of pipeline tasks of region i (its tiles times its
// split-K factor), |P_multi| the number of tasks the machine runs at once
// (warps per wave divided by the micro-kernel's warps), f_num the number of
// micro-kernel instances (K steps) in one task, and g_predict the
// micro-kernel's measured (or modelled) time for a task of f_num instances.
//
// Patterns (MikPoly summary, section 4: a GPU uses Patterns I and II):
//   I   one region, the whole output, one micro-kernel;
//   II  two regions cut along M (top / bottom) or N (left / right), each with
//       its own micro-kernel; the first region's cut is placed so that its
//       tasks fill whole waves, or so that it holds only full tiles.
// The search visits strategies in a fixed order and skips a strategy as soon
// as its running cost exceeds the best found so far.
//
// GB300 additions (readings, see the design notes): f_pipe also carries the
// split-K reduction traffic, and the total is floored by the algorithmic
// bytes over HBM bandwidth ("HBM bytes versus MMA cycles").
#include <algorithm>
#include <array>
#include <vector>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "mp_internal.h"
#include "mp_b2b.cuh"
#include "mp_conv.cuh"
#include "mp_grouped.cuh"

namespace mp {
namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Split-K on chip runs in clusters of S CTAs, one task each.  Measured on
// GB300: 2-3 us cheaper than through L2 for S <= 8; past 8 (non-portable
// cluster sizes) no cheaper, so only S <= 8 runs on chip.  The reduction's
// cost terms live in the handle (split_sync_us, split_bytes_factor).
constexpr int kClusterSplitMax = kClusterSplitMaxS;
// Floor of one uk step of any micro-kernel: the single MMA-issuing thread's
// per-instruction and per-stage cost (measured on GB300 with tiny tiles).
constexpr double kStepFloorUs = 0.21;
// Extra fixed time of a CTA-pair task: cluster set-up and exit, the
// leader's commits reaching the peer (measured on GB300: about 1.5 us).
constexpr double kPairFixedUs = 1.5;

struct RegionEval {
    int32_t kernel = -1;
    int32_t splits = 1;
    int32_t f_num = 0;
    int64_t f_parallel = 0;
    int64_t f_wave = 0;
    double f_pipe = 0.0;
    double cost = 0.0;
    double tail = 0.0;
    int64_t ws_floats = 0;
    bool ok = false;
};

inline int64_t slots_for(const mp_handle_s* h, const mp_kernel_desc& u) {
    int64_t s = h->hw.warps_per_wave / std::max(1, u.warps);
    return std::max<int64_t>(1, s);
}

// Split-K runs on chip when the handle's device can hold clusters of S CTAs
// and all `tasks` fit one wave of them (cluster_split_room).
inline bool split_on_chip(const mp_handle_s* h, const mp_kernel_desc& u, int64_t splits, int64_t tasks) {
    return !u.pair && splits >= 2 && splits <= h->cluster_split_max && splits <= kClusterSplitMax &&
           tasks <= cluster_split_room(h, (int)splits);
}

// g_predict(f_num) plus the split-K reduction: every task of a split tile
// writes an fp32 partial, waits for the tile's other splits (a counter round
// trip through L2), then reads 1/S of every partial -- one partial's worth.
inline double f_pipe_of(const mp_handle_s* h, const mp_kernel_desc& u, int64_t f_num, int64_t splits,
                        int64_t tasks) {
    double t = u.fixed_us + u.per_step_us * (double)f_num;
    if (splits > 1 && h->hw.l2_gbs > 0 && h->hw.num_pe > 0) {
        double tile_bytes = 4.0 * u.um * u.un;
        double pe_gbs = h->hw.l2_gbs / h->hw.num_pe;
        const int c = split_on_chip(h, u, splits, tasks) ? (int)splits : 0;
        t += h->split_sync_us[c] + h->split_bytes_factor[c] * tile_bytes / (pe_gbs * 1e3);  // bytes / (GB/s) -> us
    }
    return t;
}

RegionEval eval_region(const mp_handle_s* h, int32_t k, int64_t m_ext, int64_t n_ext, int64_t K,
                       int64_t batch, int32_t splits_req) {
    RegionEval r;
    const mp_kernel_desc& u = h->kernels[k];
    int64_t tiles = cdiv(m_ext, u.um) * cdiv(n_ext, u.un) * batch;
    int64_t kb = cdiv(K, u.uk);
    int64_t splits = 1, f_num = kb;
    if (kb > 0 && splits_req > 1) {
        f_num = cdiv(kb, std::min<int64_t>(splits_req, kb));
        splits = cdiv(kb, f_num);  // no empty split
    }
    r.kernel = k;
    r.splits = (int32_t)splits;
    r.f_num = (int32_t)f_num;
    r.f_parallel = tiles * splits;
    r.f_wave = cdiv(r.f_parallel, slots_for(h, u));
    r.f_pipe = f_pipe_of(h, u, f_num, splits, r.f_parallel);
    r.cost = (double)r.f_wave * r.f_pipe;
    r.tail = u.tail_us;
    r.ws_floats = splits > 1 ? tiles * splits * (int64_t)u.um * u.un : 0;
    r.ok = splits == 1 || (!u.pair && r.ws_floats <= h->workspace_floats && tiles <= kMaxCounters);
    return r;
}

// Split-K candidates for a region of `tiles` tiles: none, and the factors
// that bring the task count to about one or two waves.
int split_candidates(const mp_handle_s* h, const mp_kernel_desc& u, int64_t tiles, int64_t kb,
                     int32_t* out) {
    int n = 0;
    out[n++] = 1;
    if (kb <= 1 || tiles <= 0 || u.pair) return n;  // CTA pairs do not split K
    int64_t slots = slots_for(h, u);
    if (tiles >= slots) return n;
    static const int32_t kFactors[] = {2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64};
    for (int32_t s : kFactors) {
        if (s > kb) break;
        if (tiles * s > 2 * slots) break;
        out[n++] = s;
    }
    int64_t fill = std::min<int64_t>(kb, std::max<int64_t>(1, slots / tiles));
    if (fill > 1) out[n++] = (int32_t)fill;
    // The largest on-chip split that one wave of clusters holds.
    for (int32_t s = std::min<int32_t>(kClusterSplitMax, h->cluster_split_max); s >= 2; s--) {
        if (s <= kb && tiles * s <= cluster_split_room(h, s)) {
            out[n++] = s;
            break;
        }
    }
    return n;
}

struct Strategy {
    int32_t pattern = 0;
    int32_t nreg = 0;
    int64_t m0[2], n0[2], m_ext[2], n_ext[2];
    RegionEval ev[2];
    double sum = 0.0;   // sum of f_wave * f_pipe, plus the tail
    double cost = 0.0;  // max(sum, HBM floor)
};

// Sum of f_wave * f_pipe over the regions, plus the strategy's tail.
inline double strategy_sum(const Strategy& s) {
    double sum = 0.0, tail = 0.0;
    for (int i = 0; i < s.nreg; i++) {
        sum += s.ev[i].cost;
        tail = std::max(tail, s.ev[i].tail);
    }
    return sum + tail;
}

inline double tile_area(const mp_handle_s* h, const Strategy& s) {
    double a = 0.0;
    for (int i = 0; i < s.nreg; i++) {
        const mp_kernel_desc& u = h->kernels[s.ev[i].kernel];
        a += (double)u.um * u.un * (double)(s.m_ext[i] * s.n_ext[i]);
    }
    return a;
}

// Is `c` better than `b`?  Costs within 0.5% tie; ties go to fewer regions,
// then to the smaller work sum (more slack under the HBM floor), then to
// larger tiles, then to less split-K.
bool better(const mp_handle_s* h, const Strategy& c, const Strategy& b) {
    if (b.nreg == 0) return true;
    double tol = 0.005 * std::max(c.cost, b.cost);
    if (c.cost < b.cost - tol) return true;
    if (c.cost > b.cost + tol) return false;
    if (c.nreg != b.nreg) return c.nreg < b.nreg;
    // The ablation models break ties without the full model's work sum.
    if (h->plan_mode == MP_PLAN_MIKPOLY && std::fabs(c.sum - b.sum) > 0.005 * std::max(c.sum, b.sum))
        return c.sum < b.sum;
    double ta = tile_area(h, c), tb = tile_area(h, b);
    if (ta != tb) return ta > tb;
    int sc = 0, sb = 0;
    for (int i = 0; i < c.nreg; i++) sc += c.ev[i].splits;
    for (int i = 0; i < b.nreg; i++) sb += b.ev[i].splits;
    return sc < sb;
}

double hbm_floor_us(const mp_handle_s* h, int64_t batch, int64_t M, int64_t N, int64_t K, bool beta_c) {
    if (h->hw.hbm_gbs <= 0) return 0.0;
    double bytes = 2.0 * M * K + 2.0 * K * N + 4.0 * M * N + (beta_c ? 4.0 * M * N : 0.0);
    return bytes * (double)batch / (h->hw.hbm_gbs * 1e3);
}

// The strategy's cost under the handle's model (s.sum already holds the sum
// of f_wave * f_pipe over its regions).
double strategy_cost(const mp_handle_s* h, const Strategy& s, double floor_us) {
    double c = 0.0;
    switch (h->plan_mode) {
        case MP_PLAN_WAVE:
            for (int i = 0; i < s.nreg; i++) c += (double)s.ev[i].f_wave;
            return c;
        case MP_PLAN_PIPE:
            for (int i = 0; i < s.nreg; i++) c += s.ev[i].f_pipe;
            return c;
        default:
            return std::max(s.sum, floor_us);
    }
}

void fill_info(const mp_handle_s* h, const Strategy& s, int64_t K, mp_plan_info* out, int evaluated,
               int pruned) {
    std::memset(out, 0, sizeof(*out));
    out->pattern = s.pattern;
    out->num_regions = s.nreg;
    out->cost_us = s.cost;
    out->evaluated = evaluated;
    out->pruned = pruned;
    for (int i = 0; i < s.nreg; i++) {
        const RegionEval& e = s.ev[i];
        const mp_kernel_desc& u = h->kernels[e.kernel];
        mp_region_info& r = out->region[i];
        r.kernel = e.kernel;
        r.um = u.um; r.un = u.un; r.uk = u.uk; r.swap = u.swap; r.pair = u.pair;
        r.m0 = s.m0[i]; r.n0 = s.n0[i]; r.m_ext = s.m_ext[i]; r.n_ext = s.n_ext[i];
        r.splits = e.splits;
        r.f_num = e.f_num;
        r.f_parallel = e.f_parallel;
        r.f_wave = e.f_wave;
        r.f_pipe_us = e.f_pipe;
        out->total_tasks += e.f_parallel;
        out->workspace_bytes += 4 * e.ws_floats;
    }
    (void)K;
}

mp_status search(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K, mp_plan_info* out) {
    const double floor_us = hbm_floor_us(h, batch, M, N, K, false);
    Strategy best;
    int evaluated = 0, pruned = 0;
    // Pruning compares partial MikPoly costs, so it runs under that model only.
    const bool prune = h->plan_mode == MP_PLAN_MIKPOLY;
    auto finish = [&](Strategy& s) {
        s.sum = strategy_sum(s);
        s.cost = strategy_cost(h, s, floor_us);
        evaluated++;
        if (better(h, s, best)) best = s;
    };

    // ---- Pattern I: one micro-kernel over the whole output -------------------
    double single_cost[MP_MAX_KERNELS];
    for (int32_t k = 0; k < h->num_kernels; k++) {
        single_cost[k] = INFINITY;
        if (h->force_kernel >= 0 && k != h->force_kernel) continue;
        const mp_kernel_desc& u = h->kernels[k];
        int64_t tiles = cdiv(M, u.um) * cdiv(N, u.un) * batch;
        int32_t cands[16];
        int nc;
        if (h->force_splits > 0) {
            cands[0] = h->force_splits;
            nc = 1;
        } else {
            nc = split_candidates(h, u, tiles, cdiv(K, u.uk), cands);
        }
        for (int c = 0; c < nc; c++) {
            RegionEval e = eval_region(h, k, M, N, K, batch, cands[c]);
            if (!e.ok) { pruned++; continue; }
            Strategy s;
            s.pattern = 1;
            s.nreg = 1;
            s.m0[0] = 0; s.n0[0] = 0; s.m_ext[0] = M; s.n_ext[0] = N;
            s.ev[0] = e;
            finish(s);
            single_cost[k] = std::min(single_cost[k], e.cost + e.tail);
        }
    }
    if (h->force_kernel >= 0 || h->force_splits > 0) {
        if (best.nreg == 0) return MP_ERR_PLAN;
        fill_info(h, best, K, out, evaluated, pruned);
        return MP_OK;
    }

    // ---- Pattern II: two regions cut along M or along N ----------------------
    // First-region kernels: the three best single-kernel choices.
    // (A stable selection of the three cheapest: ties keep kernel order.)
    int32_t order[3];
    const int n_first = std::min<int32_t>(3, h->num_kernels);
    for (int i = 0; i < n_first; i++) {
        int32_t pick = -1;
        for (int32_t k = 0; k < h->num_kernels; k++) {
            bool taken = false;
            for (int j = 0; j < i; j++) taken |= order[j] == k;
            if (!taken && (pick < 0 || single_cost[k] < single_cost[pick])) pick = k;
        }
        order[i] = pick;
    }

    for (int dir = 0; dir < 2; dir++) {  // 0: cut along M, 1: cut along N
        const int64_t along = dir == 0 ? M : N;
        const int64_t across = dir == 0 ? N : M;
        for (int ia = 0; ia < n_first; ia++) {
            const int32_t a = order[ia];
            if (!std::isfinite(single_cost[a])) continue;
            const mp_kernel_desc& ua = h->kernels[a];
            const int64_t step = dir == 0 ? ua.um : ua.un;
            const int64_t blocks_across = cdiv(across, dir == 0 ? ua.un : ua.um) * batch;
            const int64_t slots = slots_for(h, ua);
            const int64_t total_blocks = cdiv(along, step);
            // Cut candidates (in blocks of the first kernel): whole waves, and
            // the largest cut that keeps only full tiles in the first region.
            int64_t cuts[8];
            int ncut = 0;
            const int64_t waves = cdiv(total_blocks * blocks_across, slots);
            for (int64_t w = 1; w < waves && ncut < 6; w++) {
                int64_t blocks = (w * slots) / blocks_across;
                if (blocks >= 1 && blocks < total_blocks) cuts[ncut++] = blocks;
            }
            if (along % step != 0 && along / step >= 1) cuts[ncut++] = along / step;
            for (int ic = 0; ic < ncut; ic++) {
                const int64_t cut = cuts[ic] * step;
                if (cut <= 0 || cut >= along) continue;
                // First region: no split (its tasks fill whole waves).
                RegionEval ea = dir == 0 ? eval_region(h, a, cut, N, K, batch, 1)
                                         : eval_region(h, a, M, cut, K, batch, 1);
                if (!ea.ok) continue;
                if (prune && std::max(ea.cost, floor_us) > best.cost * 1.005) { pruned++; continue; }
                const int64_t rest = along - cut;
                for (int32_t b = 0; b < h->num_kernels; b++) {
                    const mp_kernel_desc& ub = h->kernels[b];
                    if (dir == 1 && ub.un % 8 != 0) continue;
                    if (ub.pair != ua.pair) continue;  // one launch: all pairs or none
                    int64_t rm = dir == 0 ? rest : M, rn = dir == 0 ? N : rest;
                    int64_t tiles_b = cdiv(rm, ub.um) * cdiv(rn, ub.un) * batch;
                    int64_t kb = cdiv(K, ub.uk);
                    int32_t sb[2] = {1, 1};
                    int nsb = 1;
                    int64_t sl = slots_for(h, ub);
                    if (tiles_b < sl && kb > 1) {
                        sb[1] = (int32_t)std::min<int64_t>(kb, std::max<int64_t>(1, sl / tiles_b));
                        if (sb[1] > 1) nsb = 2;
                    }
                    for (int is = 0; is < nsb; is++) {
                        RegionEval eb = eval_region(h, b, rm, rn, K, batch, sb[is]);
                        if (!eb.ok) { pruned++; continue; }
                        if (prune && std::max(ea.cost + eb.cost, floor_us) > best.cost * 1.005) {
                            pruned++;
                            continue;
                        }
                        Strategy s;
                        s.pattern = 2;
                        s.nreg = 2;
                        if (dir == 0) {
                            s.m0[0] = 0; s.n0[0] = 0; s.m_ext[0] = cut; s.n_ext[0] = N;
                            s.m0[1] = cut; s.n0[1] = 0; s.m_ext[1] = rest; s.n_ext[1] = N;
                        } else {
                            s.m0[0] = 0; s.n0[0] = 0; s.m_ext[0] = M; s.n_ext[0] = cut;
                            s.m0[1] = 0; s.n0[1] = cut; s.m_ext[1] = M; s.n_ext[1] = rest;
                        }
                        s.ev[0] = ea;
                        s.ev[1] = eb;
                        finish(s);
                    }
                }
            }
        }
    }
    if (best.nreg == 0) return MP_ERR_PLAN;
    fill_info(h, best, K, out, evaluated, pruned);
    return MP_OK;
}

inline size_t cache_slot(const PlanKey& k, size_t n) {
    uint64_t x = (uint64_t)k.M * 0x9E3779B97F4A7C15ull ^ (uint64_t)k.N * 0xC2B2AE3D27D4EB4Full ^
                 (uint64_t)k.K * 0x165667B19E3779F9ull ^ (uint64_t)k.batch * 0x27D4EB2F165667C5ull;
    x ^= x >> 29;
    return (size_t)(x % n);
}

}  // namespace

void clear_plan_cache(mp_handle h) {
    for (auto& e : h->cache) e.key = PlanKey{-1, -1, -1, -1};
}

mp_status enumerate_plans(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                          std::vector<mp_plan_info>* out) {
    out->clear();
    if (!h || batch < 1 || M < 1 || N < 1 || K < 0) return MP_ERR_INVALID_ARG;
    const double floor_us = hbm_floor_us(h, batch, M, N, K, false);
    std::vector<Strategy> all;
    auto add = [&](Strategy& st) {
        st.sum = strategy_sum(st);
        st.cost = strategy_cost(h, st, floor_us);
        all.push_back(st);
    };

    // Pattern I: every micro-kernel with every split-K candidate.
    for (int32_t k = 0; k < h->num_kernels; k++) {
        const mp_kernel_desc& u = h->kernels[k];
        const int64_t tiles = cdiv(M, u.um) * cdiv(N, u.un) * batch;
        int32_t cands[16];
        const int nc = split_candidates(h, u, tiles, cdiv(K, u.uk), cands);
        for (int c = 0; c < nc; c++) {
            RegionEval e = eval_region(h, k, M, N, K, batch, cands[c]);
            if (!e.ok) continue;
            Strategy st;
            st.pattern = 1;
            st.nreg = 1;
            st.m0[0] = 0; st.n0[0] = 0; st.m_ext[0] = M; st.n_ext[0] = N;
            st.ev[0] = e;
            add(st);
        }
    }

    // Pattern II: two regions cut along M or along N.
    for (int dir = 0; dir < 2; dir++) {
        const int64_t along = dir == 0 ? M : N;
        const int64_t across = dir == 0 ? N : M;
        for (int32_t a = 0; a < h->num_kernels; a++) {
            const mp_kernel_desc& ua = h->kernels[a];
            const int64_t step = dir == 0 ? ua.um : ua.un;
            const int64_t total_blocks = cdiv(along, step);
            if (total_blocks < 2) continue;
            const int64_t blocks_across = cdiv(across, dir == 0 ? ua.un : ua.um) * batch;
            const int64_t slots = slots_for(h, ua);
            std::vector<int64_t> cuts;
            if (total_blocks - 1 <= 64) {
                for (int64_t c = 1; c < total_blocks; c++) cuts.push_back(c);
            } else {
                for (int i = 1; i <= 64; i++) cuts.push_back(std::max<int64_t>(1, (total_blocks - 1) * i / 65));
                const int64_t waves = cdiv(total_blocks * blocks_across, slots);
                for (int64_t w = 1; w < waves; w++) cuts.push_back((w * slots) / blocks_across);
                if (along % step != 0) cuts.push_back(along / step);
                std::sort(cuts.begin(), cuts.end());
                cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());
            }
            for (int64_t cb : cuts) {
                const int64_t cut = cb * step;
                if (cut <= 0 || cut >= along) continue;
                RegionEval ea = dir == 0 ? eval_region(h, a, cut, N, K, batch, 1) : eval_region(h, a, M, cut, K, batch, 1);
                if (!ea.ok) continue;
                const int64_t rest = along - cut;
                for (int32_t b = 0; b < h->num_kernels; b++) {
                    const mp_kernel_desc& ub = h->kernels[b];
                    if (dir == 1 && ub.un % 8 != 0) continue;
                    if (ub.pair != ua.pair) continue;
                    const int64_t rm = dir == 0 ? rest : M, rn = dir == 0 ? N : rest;
                    const int64_t tiles_b = cdiv(rm, ub.um) * cdiv(rn, ub.un) * batch;
                    const int64_t kb = cdiv(K, ub.uk);
                    int32_t sb[2] = {1, 1};
                    int nsb = 1;
                    const int64_t sl = slots_for(h, ub);
                    if (!ub.pair && tiles_b < sl && kb > 1) {
                        sb[1] = (int32_t)std::min<int64_t>(kb, std::max<int64_t>(1, sl / tiles_b));
                        if (sb[1] > 1) nsb = 2;
                    }
                    for (int is = 0; is < nsb; is++) {
                        RegionEval eb = eval_region(h, b, rm, rn, K, batch, sb[is]);
                        if (!eb.ok) continue;
                        Strategy st;
                        st.pattern = 2;
                        st.nreg = 2;
                        if (dir == 0) {
                            st.m0[0] = 0; st.n0[0] = 0; st.m_ext[0] = cut; st.n_ext[0] = N;
                            st.m0[1] = cut; st.n0[1] = 0; st.m_ext[1] = rest; st.n_ext[1] = N;
                        } else {
                            st.m0[0] = 0; st.n0[0] = 0; st.m_ext[0] = M; st.n_ext[0] = cut;
                            st.m0[1] = 0; st.n0[1] = cut; st.m_ext[1] = M; st.n_ext[1] = rest;
                        }
                        st.ev[0] = ea;
                        st.ev[1] = eb;
                        add(st);
                    }
                }
            }
        }
    }
    std::stable_sort(all.begin(), all.end(), [](const Strategy& x, const Strategy& y) { return x.cost < y.cost; });
    out->resize(all.size());
    for (size_t i = 0; i < all.size(); i++) fill_info(h, all[i], K, &(*out)[i], (int)all.size(), 0);
    return MP_OK;
}

mp_status plan_shape(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K, mp_plan_info* out) {
    if (!h || !out) return MP_ERR_INVALID_ARG;
    if (batch < 0 || M < 0 || N < 0 || K < 0) return MP_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || batch == 0) {
        std::memset(out, 0, sizeof(*out));
        out->pattern = 1;
        return MP_OK;
    }
    PlanKey key{batch, M, N, K};
    if (!h->cache.empty()) {
        PlanCacheEntry& e = h->cache[cache_slot(key, h->cache.size())];
        if (e.key == key) {
            *out = e.plan;
            return MP_OK;
        }
    }
    mp_status st = search(h, batch, M, N, K, out);
    if (st != MP_OK) return st;
    st = validate_plan(*out, M, N, K);
    if (st != MP_OK) return st;
    if (!h->cache.empty()) {
        PlanCacheEntry& e = h->cache[cache_slot(key, h->cache.size())];
        e.key = key;
        e.plan = *out;
    }
    return MP_OK;
}

mp_status validate_plan(const mp_plan_info& p, int64_t M, int64_t N, int64_t K) {
    (void)K;
    if (p.num_regions < 1 || p.num_regions > MP_MAX_REGIONS) return MP_ERR_PLAN;
    int64_t area = 0;
    for (int i = 0; i < p.num_regions; i++) {
        const mp_region_info& r = p.region[i];
        if (r.m_ext <= 0 || r.n_ext <= 0 || r.m0 < 0 || r.n0 < 0) return MP_ERR_PLAN;
        if (r.m0 + r.m_ext > M || r.n0 + r.n_ext > N) return MP_ERR_PLAN;
        if (r.n0 % 8 != 0) return MP_ERR_PLAN;  // TMA x coordinate rule on B
        if (r.splits < 1) return MP_ERR_PLAN;
        if (r.pair != p.region[0].pair || (r.pair && r.splits != 1)) return MP_ERR_PLAN;
        area += r.m_ext * r.n_ext;
        for (int j = 0; j < i; j++) {
            const mp_region_info& q = p.region[j];
            bool apart = r.m0 >= q.m0 + q.m_ext || q.m0 >= r.m0 + r.m_ext ||
                         r.n0 >= q.n0 + q.n_ext || q.n0 >= r.n0 + r.n_ext;
            if (!apart) return MP_ERR_PLAN;
        }
    }
    return area == M * N ? MP_OK : MP_ERR_PLAN;
}

mp_status evaluate_plan(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                        mp_plan_info* p) {
    if (!h || !p || batch < 1 || M < 1 || N < 1 || K < 0) return MP_ERR_INVALID_ARG;
    if (p->num_regions < 1 || p->num_regions > MP_MAX_REGIONS) return MP_ERR_INVALID_ARG;
    double sum = 0.0, tail = 0.0;
    p->total_tasks = 0;
    p->workspace_bytes = 0;
    for (int i = 0; i < p->num_regions; i++) {
        mp_region_info& r = p->region[i];
        if (r.kernel < 0 || r.kernel >= h->num_kernels) return MP_ERR_INVALID_ARG;
        RegionEval e = eval_region(h, r.kernel, r.m_ext, r.n_ext, K, batch, std::max(1, r.splits));
        const mp_kernel_desc& u = h->kernels[r.kernel];
        r.um = u.um; r.un = u.un; r.uk = u.uk; r.swap = u.swap; r.pair = u.pair;
        r.splits = e.splits;
        r.f_num = e.f_num;
        r.f_parallel = e.f_parallel;
        r.f_wave = e.f_wave;
        r.f_pipe_us = e.f_pipe;
        sum += e.cost;
        tail = std::max(tail, e.tail);
        p->total_tasks += e.f_parallel;
        p->workspace_bytes += 4 * e.ws_floats;
    }
    p->cost_us = std::max(sum + tail, hbm_floor_us(h, batch, M, N, K, false));
    if (p->pattern == 0) p->pattern = p->num_regions == 1 ? 1 : 2;
    return validate_plan(*p, M, N, K);
}

// The GB300 micro-kernel set and its analytic g_predict (used until a
// calibration table replaces it).  Normal kernels: a 128-row accumulator
// (UMMA M = 128) against un = 64..256 columns of B.  Swapped kernels compute
// D^T = B^T A^T: the UMMA M = 128 runs over N and the short M becomes the
// UMMA N (16..128), so a skinny M wastes no tensor-core rows.  Pair kernels
// put a 256-row tile on two SMs (pair MMA): each SM loads 128 rows of A and
// half of B's columns, so operand bytes per MMA fall by a third (256 wide),
// by 30% (192 wide) or by a quarter (128 wide); a task holds two SMs, and the
// cluster set-up and exit cost a fixed extra.
void default_gb300_kernels(const mp_hw& hw, mp_kernel_desc* out, int32_t* n) {
    struct G { int um, un, swap, pair; };
    static const G kSet[] = {
        {128, 256, 0, 0}, {128, 192, 0, 0}, {128, 128, 0, 0}, {128, 64, 0, 0},
        {16, 128, 1, 0},  {32, 128, 1, 0},  {64, 128, 1, 0},  {128, 128, 1, 0},
        {256, 256, 0, 1}, {256, 128, 0, 1}, {256, 192, 0, 1},
    };
    const double pe = std::max(1, hw.num_pe);
    const double mma_pe = hw.mma_tflops > 0 ? hw.mma_tflops / pe : 13.0;   // TFLOP/s per PE
    const double l2_pe = hw.l2_gbs > 0 ? hw.l2_gbs / pe : 120.0;          // GB/s per PE
    const double hbm_pe = hw.hbm_gbs > 0 ? hw.hbm_gbs / pe : 45.0;
    // The 256 x 192 pair joins the set only with MP_PAIR192=1.  Measured on
    // GB300 against the set without it (the same box, back to back): it runs
    // its K loop about 10% faster than the one-CTA 128 x 192 tile on the
    // (3520..4032, 768, 3072) GEMMs that the model gives it, yet the
    // dynamic-sequence step is 2% slower with it (0.887 against 0.869 ms), and
    // the stress and merged workloads are even.
    const char* p192 = std::getenv("MP_PAIR192");
    const bool with_192 = p192 && p192[0] == '1';
    int32_t c = 0;
    for (const G& g : kSet) {
        if (g.pair && g.un == 192 && !with_192) continue;
        mp_kernel_desc& d = out[c++];
        d.um = g.um;
        d.un = g.un;
        d.uk = kUk;
        d.warps = kModelWarpsPerTask * (g.pair ? 2 : 1);  // one CTA per SM: one task slot per PE
        d.swap = g.swap;
        d.pair = g.pair;
        // Per SM: a 128-row accumulator; a pair's SM holds half of B.
        const double n_umma = g.swap ? g.um : g.un;
        const double flops = 2.0 * kUmmaM * std::max(32.0, n_umma) * kUk;
        const double mma_us = flops / (mma_pe * 1e6);
        const double bytes = (kUmmaM + (g.pair ? n_umma / 2 : n_umma)) * kUk * 2.0;
        const double load_us = bytes / (l2_pe * 1e3);
        d.per_step_us = std::max(std::max(mma_us, load_us), kStepFloorUs);
        // Epilogue: the tile's fp32 output at the SM's share of HBM; the
        // swapped form stores straight from registers at about half the rate.
        // It is charged in every task, not once as a tail: measured on
        // GB300, a second wave costs its K loop plus most of an epilogue
        // (the first wave's stores slow the second wave's operand loads), and
        // planning with the epilogue as a once-per-plan tail made the
        // dynamic-sequence, merged-QKV and stress steps 0-5% slower.
        const double epi_bytes = 4.0 * kUmmaM * (g.swap ? g.um : g.un);  // per SM
        d.fixed_us = 0.6 + (g.swap ? 2.0 : 1.0) * epi_bytes / (hbm_pe * 1e3) + (g.pair ? kPairFixedUs : 0.0);
        d.tail_us = 0.0;
    }
    *n = c;
}

// ---------------------------------------------------------------------------
// Back-to-back GEMMs (BOLT summary, persistent kernel (GEMM/Conv) fusion)
// ---------------------------------------------------------------------------
// Work unit: 128 rows x `cpg` chunks of D1.  Each unit runs the first GEMM
// for its rows (nk0 K steps of a 128 x n0p tile), then cpg chunks of the
// second (nk1 = n0p / 64 K steps of a 128 x bn1 tile, each followed by its
// fp32 epilogue; a chunk's epilogue overlaps the next chunk's MMAs, and a
// unit's last epilogue the next unit's first GEMM).  Fewer
// chunks per unit give more units to spread over the SMs, at the price of
// recomputing the block of D0 once per unit.
mp_status plan_b2b(const mp_hw& hw, int64_t M, int64_t N0, int64_t N1, int64_t K0, mp_b2b_plan* out) {
    if (!out || M < 0 || N0 < 0 || N1 < 0 || K0 < 0) return MP_ERR_INVALID_ARG;
    if (N0 > 256) return MP_ERR_UNSUPPORTED;
    if (M >= ((int64_t)1 << 31) || N1 >= ((int64_t)1 << 31) || K0 >= ((int64_t)1 << 31)) return MP_ERR_INVALID_ARG;
    const int64_t k0 = N0 > 0 ? K0 : 0;  // no first GEMM without columns of D0
    const int n0p = (int)(((N0 + 63) / 64) * 64);
    const int nk0 = (int)((k0 + 63) / 64), nk1 = n0p / 64;
    const int mblocks = (int)((M + 127) / 128);
    const int sms = std::max(1, hw.num_pe);
    const double hbm = hw.hbm_gbs > 0 ? hw.hbm_gbs : 6700.0;
    // Phase times of one unit, measured on GB300 with timestamped copies of
    // the kernel: a 64-deep K step of a 128 x n tile costs about 0.40 us at
    // n = 256 (operand ingest and the MMA issuer), never below the issuer's
    // floor; the hand-over of D0 about 0.3 us + 0.9 us per 256 columns; a
    // chunk's epilogue about 1.6 us per 256 columns when its stores are not
    // HBM-bound; the first operands of a CTA arrive after about 1 us.
    auto step_us = [&](int n) { return std::max(kStepFloorUs, 0.40 * n / 256.0); };
    const double handover = 0.3 + 0.9 * n0p / 256.0;
    const double t0 = nk0 * (n0p > 0 ? step_us(n0p) : 0.0) + handover;
    mp_b2b_plan best;
    std::memset(&best, 0, sizeof best);
    best.cost_us = 1e300;
    const int widest = (int)std::min<int64_t>(256, std::max<int64_t>(64, ((N1 + 63) / 64) * 64));
    // Chunk width: the widest tile that covers N1 (up to 256), or 128 (twice
    // the units per row block, each chunk's MMAs and stores half as long).
    const int widths[2] = {widest, widest > 128 ? 128 : 0};
    for (int bn1 : widths) {
        if (bn1 == 0) continue;
        const int chunks = (int)((N1 + bn1 - 1) / bn1);
        const int stage_bytes = std::max(nk0 > 0 ? 16384 + n0p * 128 : 0, bn1 * 128);
        const int room = b2b::kSmemLimit - n0p * 256 - 4 * b2b::kEpiSlabBytes - 2048;
        const int stages = std::min(b2b::kMaxStages, room / stage_bytes);
        if (stages < 2) continue;
        const double mma1 = nk1 * step_us(bn1);
        for (int cpg = 1; cpg <= std::max(1, chunks); cpg++) {
            const int64_t groups = (chunks + cpg - 1) / cpg;
            if (cpg > 1 && (chunks + cpg - 2) / (cpg - 1) == groups) continue;  // same grouping as cpg - 1
            const int64_t units = (int64_t)mblocks * std::max<int64_t>(1, groups);
            const int64_t active = std::min<int64_t>(units, sms);
            // A chunk's fp32 output at the active SMs' share of HBM bandwidth,
            // or the epilogue warps' own rate, whichever is slower.
            const double hbm_pe = hbm * 1e3 / (double)active;  // bytes per us per active SM
            const double epi = std::max(1.6 * bn1 / 256.0, 4.0 * 128 * bn1 / hbm_pe);
            // The block of A0 comes from HBM once per row block (the units of a
            // row block run side by side), so each unit carries 1/groups of it.
            const double a0_us = 2.0 * 128 * (double)k0 / (double)std::max<int64_t>(1, groups) / hbm_pe;
            // A CTA's units form a pipeline: the MMA side (first GEMM, hand-over,
            // the chunks' MMAs) of one unit overlaps the epilogue warps' side
            // (hand-over, the chunks' stores, and the unit's share of HBM
            // traffic) of the one before, so each unit costs the slower side,
            // plus one fill/drain.
            const double mma_side = t0 + cpg * mma1;
            const double epi_side = handover + std::max(cpg * epi, a0_us + cpg * 4.0 * 128 * bn1 / hbm_pe);
            const double waves = (double)((units + sms - 1) / sms);
            const double cost = 1.0 + waves * std::max(mma_side, epi_side) + std::min(mma_side, epi_side) + 2.0;
            if (cost < best.cost_us * (1.0 - 1e-9)) {
                best.cost_us = cost;
                best.n0p = n0p;
                best.bn1 = bn1;
                best.chunks = chunks;
                best.mblocks = mblocks;
                best.cpg = cpg;
                best.units = (int32_t)units;
                best.num_stages = stages;
                best.stage_bytes = stage_bytes;
            }
        }
    }
    if (best.bn1 == 0) return MP_ERR_PLAN;
    best.grid = (int32_t)std::min<int64_t>(best.units, sms);
    best.smem_bytes = b2b::smem_bytes(best.num_stages, best.stage_bytes, best.n0p);
    *out = best;
    return MP_OK;
}

// ---------------------------------------------------------------------------
// Implicit-GEMM convolution (MikPoly summary, section 5: convolutions as GEMM)
// ---------------------------------------------------------------------------
// The GEMM's M runs over output pixels, cut into boxes of wb x hb x nb
// (along Q, P and images; powers of two, product 128, one UMMA's rows); its
// N over output channels in tiles of bn; its K over filter taps x blocks of
// 64 channels.  Small images waste part of a box, so every box shape is
// tried: the cost is the waves of tiles times the slower of a tile's K loop
// and its stores (a CTA's tiles pipeline through two accumulators), plus
// one fill.  The constants are those measured for the GEMM kernels.
mp_status plan_conv(const mp_hw& hw, int64_t ws_floats, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K,
                    int64_t R, int64_t S, int64_t pad_h, int64_t pad_w, mp_conv_plan* out) {
    if (!out || N < 0 || H < 0 || W < 0 || C < 0 || K < 0 || R < 1 || S < 1 || pad_h < 0 || pad_w < 0)
        return MP_ERR_INVALID_ARG;
    const int64_t lim = (int64_t)1 << 31;
    if (N >= lim || H >= lim || W >= lim || C >= lim || K >= lim || R >= lim || S >= lim || pad_h >= lim ||
        pad_w >= lim || R * S * (C + 63) >= lim)
        return MP_ERR_INVALID_ARG;
    const int64_t P = H + 2 * pad_h - R + 1, Q = W + 2 * pad_w - S + 1;
    mp_conv_plan best;
    std::memset(&best, 0, sizeof best);
    if (N == 0 || K == 0 || P <= 0 || Q <= 0) {  // empty output
        best.wb = 128;
        best.hb = best.nb = 1;
        best.bn = 64;
        best.splits = 1;
        *out = best;
        return MP_OK;
    }
    const int sms = std::max(1, hw.num_pe);
    const double hbm = hw.hbm_gbs > 0 ? hw.hbm_gbs : 6700.0;
    const int64_t ksteps = R * S * ((C + 63) / 64);
    best.cost_us = 1e300;
    const int64_t kcover = ((K + 63) / 64) * 64;
    // A K step of this kernel (a 4-D box of X and the filter's boxes), measured
    // on GB300: about 0.6 us up to bn = 128 (operand requests, not MMAs,
    // bound it), more for the widest tile.
    auto step_us = [](int bn) { return bn <= 128 ? 0.6 : 0.8; };
    for (int bn : {64, 128, 256}) {
        if (bn > 64 && bn / 2 >= kcover) continue;  // wider than the channels need
        const int64_t tiles_k = (K + bn - 1) / bn;
        const int stage_bytes = 16384 + bn * 128;
        const int stages = std::min(conv::kMaxStages, (conv::kSmemLimit - 4 * conv::kEpiSlabBytes - 2048) / stage_bytes);
        // Box shapes: powers of two with product 128, and sides that divide
        // the output exactly (Q / k, P / k) with as many images as fit.
        std::vector<std::array<int, 3>> boxes;
        for (int wb = 1; wb <= 128; wb *= 2)
            for (int hb = 1; wb * hb <= 128; hb *= 2) boxes.push_back({wb, hb, 128 / (wb * hb)});
        for (int kq = 1; kq <= 4; kq++) {
            const int wb = (int)((Q + kq - 1) / kq);
            if (wb > 128) continue;
            for (int kp = 1; kp <= 8; kp++) {
                const int hb = (int)((P + kp - 1) / kp);
                if (wb * hb > 128) continue;
                const int nb = (int)std::min<int64_t>(N, 128 / (wb * hb));
                boxes.push_back({wb, hb, nb});
            }
        }
        for (const auto& box : boxes) {
            {
                const int wb = box[0], hb = box[1], nb = box[2];
                const bool pow2 = wb * hb * nb == 128 && !(wb & (wb - 1)) && !(hb & (hb - 1)) && !(nb & (nb - 1));
                const int64_t tq = (Q + wb - 1) / wb, tp = (P + hb - 1) / hb, tn = (N + nb - 1) / nb;
                const int64_t tiles = tq * tp * tn * tiles_k;
                const double useful = (double)(N * P * Q) / (double)(tq * wb * tp * hb * tn * nb);
                for (int splits : {1, 2, 3, 4, 6, 8, 12, 16}) {
                    if (splits > 1 && (splits > ksteps || tiles * splits * 128 * bn > ws_floats)) continue;
                    const int64_t units = tiles * splits;
                    if (units >= lim) continue;
                    const int64_t active = std::min<int64_t>(units, sms);
                    const double hbm_pe = hbm * 1e3 / (double)active;  // bytes per us per active SM
                    // Pixel-by-pixel stores (boxes that are not powers of two)
                    // take about twice as long as the warps' box stores.
                    const double epi = std::max(1.6 * bn / 256.0 * (pow2 ? 1.0 : 2.0), 4.0 * 128 * bn / hbm_pe);
                    const double mma = (double)((ksteps + splits - 1) / splits) * step_us(bn);
                    const double waves = (double)((units + sms - 1) / sms);
                    // The reduction: a second launch reading every partial once.
                    const double reduce = splits > 1 ? 3.0 + (double)(tiles * splits * 128 * bn * 4 + N * P * Q * K * 4) /
                                                               (hbm * 1e3)
                                                     : 0.0;
                    const double cost = 1.0 + waves * std::max(mma, epi) + std::min(mma, epi) + 2.0 + reduce;
                    if (cost < best.cost_us * (1.0 - 1e-9) ||
                        (cost < best.cost_us * (1.0 + 1e-9) && useful > best.useful)) {
                        best.cost_us = cost;
                        best.wb = wb;
                        best.hb = hb;
                        best.nb = nb;
                        best.bn = bn;
                        best.tiles_q = (int32_t)tq;
                        best.tiles_p = (int32_t)tp;
                        best.tiles_n = (int32_t)tn;
                        best.tiles_k = (int32_t)tiles_k;
                        best.tiles = (int32_t)tiles;
                        best.splits = splits;
                        best.units = (int32_t)units;
                        best.useful = useful;
                        best.num_stages = stages;
                        best.stage_bytes = stage_bytes;
                    }
                }
            }
        }
    }
    if (best.units == 0) return MP_ERR_PLAN;
    best.ksteps = (int32_t)ksteps;
    best.grid = (int32_t)std::min<int64_t>(best.units, sms);
    best.smem_bytes = conv::smem_bytes(best.num_stages, best.stage_bytes);
    *out = best;
    return MP_OK;
}

// ---------------------------------------------------------------------------
// Grouped GEMM (BladeDISC v0.2.0 notes, GEMM merging, any shapes)
// ---------------------------------------------------------------------------
// One micro-kernel (128 x bn) for the whole group.  Cost: the group's tile
// work spread over the SMs (or the longest tile, if that is longer), plus
// one fill and launch per 48 problems.  Step times as for the other kernels.
mp_status plan_grouped(const mp_hw& hw, int32_t count, const mp_gemm_problem* probs, mp_grouped_plan* out) {
    if (!out || count < 0 || (count > 0 && !probs)) return MP_ERR_INVALID_ARG;
    mp_grouped_plan best;
    std::memset(&best, 0, sizeof best);
    best.cost_us = 1e300;
    const int sms = std::max(1, hw.num_pe);
    const double hbm = hw.hbm_gbs > 0 ? hw.hbm_gbs : 6700.0;
    int64_t maxn = 64;
    for (int32_t i = 0; i < count; i++) maxn = std::max<int64_t>(maxn, probs[i].N);
    for (int bn : {64, 128, 256}) {
        if (bn > 64 && bn / 2 >= ((maxn + 63) / 64) * 64) continue;
        const double step = std::max(kStepFloorUs, 0.40 * bn / 256.0);
        const double epi = 1.6 * bn / 256.0;
        int64_t units = 0;
        double work = 0.0, longest = 0.0;
        for (int32_t i = 0; i < count; i++) {
            const mp_gemm_problem& q = probs[i];
            const int64_t tiles = ((q.M + 127) / 128) * ((q.N + bn - 1) / bn);
            const double t = (double)((q.K + 63) / 64) * step + epi;
            units += tiles;
            work += (double)tiles * t;
            longest = std::max(longest, t);
        }
        const int64_t active = std::max<int64_t>(1, std::min<int64_t>(units, sms));
        double bytes = 0.0;  // D of every problem, at HBM speed: the floor of a store-bound group
        for (int32_t i = 0; i < count; i++) bytes += 4.0 * (double)probs[i].M * (double)probs[i].N;
        const int launches = (count + grp::kMaxGroup - 1) / grp::kMaxGroup;
        const double cost = std::max(std::max(work / (double)active, longest), bytes / (hbm * 1e3)) + 3.0 * launches;
        if (cost < best.cost_us * (1.0 - 1e-9)) {
            best.cost_us = cost;
            best.bn = bn;
            best.units = (int32_t)std::min<int64_t>(units, ((int64_t)1 << 31) - 1);
            best.launches = launches;
            best.stage_bytes = 16384 + bn * 128;
            best.num_stages =
                std::min(grp::kMaxStages, (grp::kSmemLimit - 4 * grp::kEpiSlabBytes - 2048) / best.stage_bytes);
        }
    }
    best.smem_bytes = grp::smem_bytes(best.num_stages, best.stage_bytes);
    *out = best;
    return MP_OK;
}

}  // namespace mp
