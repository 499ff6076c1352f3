// Host-only check of the work partition used by the Based kernels (compiled with nvcc, run on
// the CPU), for many shapes and SM counts:
//  - the head lanes divide H and leave no SM idle that the one-lane partition would use, and the
//    forward CTAs, walking their ranges with the kernels' cursor, cover every (b, h, chunk) of
//    the problem exactly once;
//  - within a lane, the pieces of the aggregate pass cover every chunk of every stretch (the last
//    stretch of a range that ends inside a head) exactly once, each piece inside one head, and the
//    aggregate CTAs' loads differ by at most one chunk (or each CTA has one whole stretch, the
//    fallback);
//  - every range that starts inside a head finds in the slots it reads (after the scan, when the
//    plan runs one) exactly the chunks of its head before its first chunk, and no slot is read that
//    the aggregate pass did not write;
//  - the lead-in cut: its ranges, walked with the cursor from the start of each one's lead-in,
//    cover every (b, h, chunk) exactly once outside the lead-ins, each lead-in is the chunks of
//    its range's first head before the range, no range is longer than the cost model allows
//    (the makespan it returns), and the launch order is a permutation of the ranges, costliest
//    first.
#include <cstdio>
#include <vector>

#include "../linear_attention_gb300/csrc/based_plan.h"

using namespace based;

namespace {
AggPlan plan;  // large: kept out of the stack
Ranges lead;

// Every (b, h, c) is visited once by the CTAs' cursors.
bool lanes_cover(int B, int H, int n_c, int L, long long N, int G) {
    std::vector<unsigned char> seen(static_cast<size_t>(B) * H * n_c, 0);
    for (int x = 0; x < G * L; ++x) {
        const int j = x / L, r = x % L;
        const Part p = cta_range(N, G, j);
        Cursor cu;
        cu.init(p.g0, static_cast<int>(p.g1 - p.g0), n_c, H / L, L, r);
        for (long long g = p.g0; g < p.g1; ++g, cu.next()) {
            if (cu.b < 0 || cu.b >= B || cu.h < 0 || cu.h >= H || cu.h % L != r) return false;
            unsigned char &s = seen[(static_cast<size_t>(cu.b) * H + cu.h) * n_c + cu.c];
            if (s) return false;
            s = 1;
        }
    }
    for (unsigned char s : seen)
        if (!s) return false;
    return true;
}

// The lead-in cut R (G ranges, the first `used` non-empty, makespan M): every (b, h, c) is in
// exactly one range, every lead-in is [head start, g0) of the range's first head, and every
// range's cost is at most M.
bool lead_cover(int B, int H, int n_c, int L, long long N, int G, const Ranges &R, int used, long long M) {
    if (used < 1 || used > G || R.g0[0] != 0 || R.g0[used] != N) return false;
    for (int j = used; j <= G; ++j)
        if (R.g0[j] != N) return false;
    std::vector<unsigned char> seen(static_cast<size_t>(B) * H * n_c, 0);
    for (int x = 0; x < used * L; ++x) {
        const int j = x / L, r = x % L;
        const long long g0 = R.g0[j], g1 = R.g0[j + 1];
        const int lead_n = static_cast<int>(g0 % n_c);
        if (g1 <= g0 || !R.lead_in || R.cnt[j] != 0) return false;
        if (range_cost(lead_n, g1 - g0) > M) return false;
        Cursor cu;
        cu.init(g0 - lead_n, static_cast<int>(lead_n + g1 - g0), n_c, H / L, L, r);
        const int b0 = cu.b, h0 = cu.h;
        if (cu.c != 0 && lead_n > 0) return false;
        for (long long g = g0 - lead_n; g < g1; ++g, cu.next()) {
            if (cu.b < 0 || cu.b >= B || cu.h < 0 || cu.h >= H || cu.h % L != r) return false;
            if (g < g0) {  // lead-in: the first head, chunks 0 .. lead_n - 1
                if (cu.b != b0 || cu.h != h0 || cu.c != g - (g0 - lead_n)) return false;
                continue;
            }
            unsigned char &s = seen[(static_cast<size_t>(cu.b) * H + cu.h) * n_c + cu.c];
            if (s) return false;
            s = 1;
        }
    }
    for (unsigned char s : seen)
        if (!s) return false;
    // the launch order: a permutation of the ranges, costliest first
    std::vector<unsigned char> ord(used, 0);
    for (int i = 0; i < used; ++i) {
        if (R.order[i] >= used || ord[R.order[i]]) return false;
        ord[R.order[i]] = 1;
        if (i > 0) {
            const int a = R.order[i - 1], b = R.order[i];
            if (range_cost(R.g0[a] % n_c, R.g0[a + 1] - R.g0[a]) < range_cost(R.g0[b] % n_c, R.g0[b + 1] - R.g0[b]))
                return false;
        }
    }
    return true;
}
}  // namespace

int main() {
    long long checked = 0, balanced_plans = 0, fallback_plans = 0, scanned = 0, laned = 0, lead_cuts = 0,
              lead_chosen = 0;
    for (int sms : {1, 2, 7, 148, 152, 160, 256}) {
        for (int K : {8, 16}) {
            for (int B : {1, 3}) {
                for (int H : {1, 2, 3, 5, 12, 16, 40, 64}) {
                    for (int T : {1, 64, 127, 128, 129, 300, 1000, 3000, 4096, 16384}) {
                        // the split the library's plan uses
                        const LaneSplit ls = lane_split(B, T, H, K, sms);
                        const int n_c = ls.n_c, L = ls.L, G = ls.G;
                        const long long N = ls.N;
                        const long long n_all = 1ll * B * H * n_c;
                        if (n_c != (T + kChunk - 1) / kChunk || N * L != n_all) { printf("bad split\n"); return 1; }
                        if (L < 1 || H % L != 0 || L > 128 / (2 * K)) { printf("bad lanes\n"); return 1; }
                        if (G < 1 || G > kMaxRanges || G > N || G * L > sms) { printf("bad range count\n"); return 1; }
                        const int g1 = static_cast<int>(n_all < sms ? n_all : (sms < kMaxRanges ? sms : kMaxRanges));
                        if (G * L < g1) {
                            printf("lanes leave SMs idle: sms=%d K=%d B=%d H=%d T=%d\n", sms, K, B, H, T);
                            return 1;
                        }
                        if (!lanes_cover(B, H, n_c, L, N, G)) {
                            printf("lane cover: sms=%d K=%d B=%d H=%d T=%d L=%d\n", sms, K, B, H, T, L);
                            return 1;
                        }
                        if (L > 1) ++laned;
                        {
                            const long long M = lead_cut(N, G, n_c, lead);
                            int used = 0;
                            while (used < G && lead.g0[used + 1] > lead.g0[used]) ++used;
                            if (!lead_cover(B, H, n_c, L, N, G, lead, used, M)) {
                                printf("lead-in cut: sms=%d K=%d B=%d H=%d T=%d L=%d\n", sms, K, B, H, T, L);
                                return 1;
                            }
                            ++lead_cuts;
                        }
                        for (int max_slots : {kMaxPieces, 203, 0}) {
                            std::vector<int> covered(N, 0), in_stretch(N, 0);
                            for (int i = 0; i < G; ++i) {
                                const Part p = cta_range(N, G, i);
                                if (p.g1 <= p.g0) { printf("empty range\n"); return 1; }
                                for (long long g = p.g0; g < p.g1; ++g) covered[g]++;
                                if (has_aggregate(N, G, i, n_c)) {
                                    const long long h = (p.g1 - 1) / n_c;
                                    for (long long g = (p.g0 > h * n_c ? p.g0 : h * n_c); g < p.g1; ++g) in_stretch[g] = 1;
                                }
                            }
                            for (long long g = 0; g < N; ++g)
                                if (covered[g] != 1) { printf("chunk %lld covered %d times\n", g, covered[g]); return 1; }
                            make_agg_plan(N, G, n_c, G, max_slots, plan);
                            {
                                bool need = false;
                                for (int i = 0; i < G; ++i) need = need || has_aggregate(N, G, i, n_c);
                                Ranges chosen;
                                const int used = need ? choose_lead_in(N, G, n_c, 64, plan, chosen) : 0;
                                if (used > 0) {
                                    ++lead_chosen;
                                    if (!lead_cover(B, H, n_c, L, N, G, chosen, used, lead_cut(N, G, n_c, lead))) {
                                        printf("chosen lead-in cut\n");
                                        return 1;
                                    }
                                }
                                if (choose_lead_in(N, G, n_c, 128, plan, chosen) != 0) { printf("lead-in for V = 128\n"); return 1; }
                            }
                            const AggPieces &A = plan.pieces;
                            // pieces: inside one head and one stretch, each stretch chunk exactly once
                            std::vector<int> piece_cov(N, 0);
                            std::vector<long long> lo(A.n), hi(A.n), hd(A.n);
                            if (A.n > kMaxPieces) { printf("too many pieces\n"); return 1; }
                            for (int q = 0; q < A.n; ++q) {
                                lo[q] = A.g0[q];
                                hi[q] = A.g0[q] + A.len[q];
                                hd[q] = lo[q] / n_c;
                                if (A.len[q] <= 0 || (hi[q] - 1) / n_c != hd[q]) { printf("bad piece\n"); return 1; }
                                for (long long g = lo[q]; g < hi[q]; ++g) piece_cov[g]++;
                            }
                            for (long long g = 0; g < N; ++g)
                                if (piece_cov[g] != in_stretch[g]) { printf("stretch chunk %lld in %d pieces\n", g, piece_cov[g]); return 1; }
                            // CTAs: consecutive pieces, balanced loads (or one stretch each)
                            if (A.cta_first[0] != 0 || A.cta_first[A.n_cta] != A.n) { printf("bad CTA pieces\n"); return 1; }
                            if (A.n_cta > G) { printf("more aggregate CTAs than ranges\n"); return 1; }
                            long long mn = N, mx = 0;
                            for (int j = 0; j < A.n_cta; ++j) {
                                long long load = 0;
                                if (A.cta_first[j + 1] <= A.cta_first[j]) { printf("CTA without pieces\n"); return 1; }
                                for (int q = A.cta_first[j]; q < A.cta_first[j + 1]; ++q) load += A.len[q];
                                mn = load < mn ? load : mn;
                                mx = load > mx ? load : mx;
                            }
                            if (A.n_cta > 0) {
                                if (mx - mn <= 1) ++balanced_plans;
                                else if (A.n == A.n_cta) ++fallback_plans;
                                else { printf("unbalanced plan\n"); return 1; }
                            }
                            if (A.n > max_slots && A.n != A.n_cta) { printf("slot budget exceeded\n"); return 1; }
                            // scan over the listed runs: slot q takes the chunks of slot q-1
                            if (plan.scan) {
                                ++scanned;
                                for (int r = 0; r < plan.runs.n; ++r) {
                                    const int q0 = plan.runs.start[r], len = plan.runs.len[r];
                                    if (len < 2 || q0 + len > A.n) { printf("bad run\n"); return 1; }
                                    for (int q = q0 + 1; q < q0 + len; ++q) {
                                        if (hd[q] != hd[q - 1] || hi[q - 1] != lo[q]) { printf("bad run link\n"); return 1; }
                                        lo[q] = lo[q - 1];
                                    }
                                }
                            }
                            // prefixes
                            for (int i = 0; i < G; ++i) {
                                const Part p = cta_range(N, G, i);
                                const int cnt = plan.pre.cnt[i];
                                if (p.g0 % n_c == 0) {
                                    if (cnt != 0) { printf("prefix at a head start\n"); return 1; }
                                    continue;
                                }
                                if (cnt < 1 || (plan.scan ? cnt != 1 : cnt > kMaxChain)) { printf("bad prefix count\n"); return 1; }
                                const int q0 = plan.pre.slot[i];
                                if (q0 + cnt > A.n) { printf("prefix reads an unwritten slot\n"); return 1; }
                                const long long h = p.g0 / n_c;
                                long long end = p.g0;
                                for (int q = q0 + cnt - 1; q >= q0; --q) {
                                    if (hd[q] != h || hi[q] != end) {
                                        printf("prefix gap: sms=%d B=%d H=%d T=%d i=%d\n", sms, B, H, T, i);
                                        return 1;
                                    }
                                    end = lo[q];
                                }
                                if (end != h * n_c) { printf("prefix short: sms=%d B=%d H=%d T=%d i=%d\n", sms, B, H, T, i); return 1; }
                                ++checked;
                            }
                        }
                    }
                }
            }
        }
    }
    printf("ok %lld prefixed ranges checked (%lld balanced plans, %lld one-stretch-per-CTA, %lld with a scan, "
           "%lld shapes with several head lanes, %lld lead-in cuts, %lld plans choose lead-ins)\n",
           checked, balanced_plans, fallback_plans, scanned, laned, lead_cuts, lead_chosen);
    return 0;
}
