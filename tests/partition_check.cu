// Host-only check of the work partition used by the Based kernels (compiled with nvcc, run on
// the CPU): for many shapes and SM counts, every chunk is covered exactly once, each range that
// starts inside a head finds exactly the chunks of that head before it, either in slot i-1 after
// the scan or, when every run is at most kMaxChain long (no scan), in the slots it sums itself,
// and no aggregate slot is read that the aggregate pass did not write.
#include <cstdio>
#include <vector>

#include "../linear_attention_gb300/csrc/based_kernels.cuh"

using namespace based;

int main() {
    long long checked = 0;
    for (int sms : {1, 2, 7, 148, 152, 160, 256}) {
        for (int heads : {1, 2, 3, 5, 16, 64, 96, 256}) {
            for (int T : {1, 64, 127, 128, 129, 300, 1000, 3000, 4096, 16384}) {
                const int n_c = (T + kChunk - 1) / kChunk;
                const long long N = 1ll * heads * n_c;
                const int G = static_cast<int>(N < sms ? N : sms);
                // slot contents as (head, first chunk, last chunk + 1) intervals
                std::vector<long long> lo(G, -1), hi(G, -1), hd(G, -1);
                std::vector<int> covered(N, 0);
                for (int i = 0; i < G; ++i) {
                    const Part p = cta_range(N, G, i);
                    if (p.g1 <= p.g0) { printf("empty range\n"); return 1; }
                    for (long long g = p.g0; g < p.g1; ++g) covered[g]++;
                    if (has_aggregate(N, G, i, n_c)) {
                        const long long h = (p.g1 - 1) / n_c;
                        const long long ga = p.g0 > h * n_c ? p.g0 : h * n_c;
                        lo[i] = ga; hi[i] = p.g1; hd[i] = h;
                    }
                }
                for (long long g = 0; g < N; ++g)
                    if (covered[g] != 1) { printf("chunk %lld covered %d times\n", g, covered[g]); return 1; }
                // without a scan: the slots a prefixed range sums are adjacent stretches of its
                // head that end at its first chunk and start at the head's first chunk
                const ScanRuns runs = make_scan_runs(N, G, n_c);
                bool scan = false;
                for (int r = 0; r < runs.n; ++r) scan = scan || runs.len[r] > kMaxChain;
                if (!scan) {
                    for (int i = 0; i < G; ++i) {
                        const Part p = cta_range(N, G, i);
                        if (p.g0 % n_c == 0) continue;
                        const long long h = p.g0 / n_c;
                        const int m = prefix_chain_len(N, G, i, n_c, kMaxChain);
                        if (m < 1 || m > kMaxChain || i - m < 0) { printf("bad chain length\n"); return 1; }
                        long long end = p.g0;
                        for (int j = i - 1; j >= i - m; --j) {
                            if (hd[j] != h || hi[j] != end) { printf("chain gap: i=%d j=%d\n", i, j); return 1; }
                            end = lo[j];
                        }
                        if (end != h * n_c) {
                            printf("chain short: sms=%d heads=%d T=%d i=%d\n", sms, heads, T, i);
                            return 1;
                        }
                        ++checked;
                    }
                }
                // scan over the runs the host lists: slot j takes the chunks of slot j-1
                for (int r = 0; r < runs.n; ++r) {
                    const int i0 = runs.start[r], len = runs.len[r];
                    if (len < 2 || i0 + len > G) { printf("bad run\n"); return 1; }
                    for (int j = i0 + 1; j < i0 + len; ++j) {
                        if (hd[j] < 0 || hd[j] != hd[j - 1] || hi[j - 1] != lo[j]) { printf("bad chain link\n"); return 1; }
                        lo[j] = lo[j - 1];
                    }
                }
                for (int i = 0; i < G; ++i) {
                    const Part p = cta_range(N, G, i);
                    if (p.g0 % n_c == 0) continue;
                    const long long h = p.g0 / n_c;
                    if (i == 0 || hd[i - 1] != h || lo[i - 1] != h * n_c || hi[i - 1] != p.g0) {
                        printf("prefix mismatch: sms=%d heads=%d T=%d i=%d\n", sms, heads, T, i);
                        return 1;
                    }
                    ++checked;
                }
            }
        }
    }
    printf("ok %lld prefixed ranges checked\n", checked);
    return 0;
}
