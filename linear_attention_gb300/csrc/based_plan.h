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

}  // namespace based
