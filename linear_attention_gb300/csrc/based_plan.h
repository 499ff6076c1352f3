// Work split of one call (host side; the partition check uses the same function): chunks per
// head, head lanes, and the chunks and ranges of one lane.
#pragma once
#include "based_kernels.cuh"

namespace based {

struct LaneSplit {
    int n_c;      // chunks per head
    int L;        // head lanes (choose_lanes); every lane has the same partition
    long long N;  // chunks of one lane
    int G;        // ranges of one lane (forward CTAs: G L)
};

// One range per SM (at most kMaxRanges per lane), or one per chunk when there are fewer chunks.
inline LaneSplit lane_split(int B, int T, int H, int K, int sms) {
    LaneSplit s;
    s.n_c = (T + kChunk - 1) / kChunk;
    const long long n_all = static_cast<long long>(B) * H * s.n_c;
    s.L = choose_lanes(K, H, n_all, sms);
    s.N = n_all / s.L;
    const int gmax = sms / s.L < kMaxRanges ? sms / s.L : kMaxRanges;
    s.G = static_cast<int>(s.N < gmax ? s.N : gmax);
    return s;
}

// Estimated makespan, in the units of the lead-in cost model (thousandths of a forward chunk), of
// the other way to give ranges their prefixes: the aggregate pass (its longest CTA load in
// chunks: agg_load), the scan when the plan needs it, the prefix loads, then the longest range of
// the even cut. Fitted to calls measured on GB300 (V = 64): about 6.8 forward chunks of fixed
// cost (launch, the aggregate pass's fill and slot writes, the prefix load and conversion) and
// 0.29 per chunk of the longest aggregate load.
constexpr long long kAggFixedCost = 6800, kAggChunkCost = 290, kScanCost = 1600;
inline long long slot_plan_cost(long long N, int G, long long agg_load, bool scan) {
    return kStartCost + kAggFixedCost + kAggChunkCost * agg_load + (scan ? kScanCost : 0) + 1000 * ((N + G - 1) / G);
}

// Lead-ins or slots (V = 64, when some range of the even cut needs a prefix): the lead-in cut of
// the lane's chunks is written to R, and it is taken when the slot plan's estimate (agg: the
// aggregate plan of the even cut) exceeds its own by kLeadMargin percent: a margin for the two
// estimates' errors (the slot plan's is a fit to measured calls, the lead-in plan's the per-CTA
// cost model). Measured on GB300 (us per call, back to back, slots / lead-ins, with the
// estimates' ratio): B2 T2048 H16 K16 23.9 / 17.9 (1.50), B1 T512 H2 K8 7.5 / 6.2 (1.68),
// B4 T4096 H16 K16 48.6 / 41.5 (1.22), B8 T16384 H32 K16 467.3 / 471.3 (1.01).
// Returns the number of ranges of the lead-in cut (the rest are empty), or 0 when the slot plan
// stays.
constexpr long long kLeadMargin = 15;
inline int choose_lead_in(long long N, int G, int n_c, int V, const AggPlan &agg, Ranges &R) {
    if (V != 64) return 0;
    const long long cost_lead = lead_cut(N, G, n_c, R);
    long long agg_load = 0;
    for (int j = 0; j < agg.pieces.n_cta; ++j) {
        long long load = 0;
        for (int q = agg.pieces.cta_first[j]; q < agg.pieces.cta_first[j + 1]; ++q) load += agg.pieces.len[q];
        agg_load = load > agg_load ? load : agg_load;
    }
    if (100 * slot_plan_cost(N, G, agg_load, agg.scan) < (100 + kLeadMargin) * cost_lead) return 0;
    int used = 0;
    while (used < G && R.g0[used + 1] > R.g0[used]) ++used;
    return used;
}

}  // namespace based
