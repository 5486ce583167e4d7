// Host-side check of the work-stealing group arithmetic (pgt_sched.cuh, WsGroups): reads
// lines "T P G layout full" from stdin and prints, per group, "g: t0 t1 ..." (its tiles in
// ticket order) when full is 1, else "g: size first last" (-1 for an empty group), then
// "end".  Compiled and compared with the oracle's group tiles by
// tests/test_ws_groups_host.py; no GPU is used.
#include <cstdio>

#include "pgt_sched.cuh"

int main() {
    int T, P, G, layout, full;
    while (std::scanf("%d %d %d %d %d", &T, &P, &G, &layout, &full) == 5) {
        pgt::WsGroups wg;
        wg.init(T, P, G, layout);
        for (int g = 0; g < G; ++g) {
            const int n = wg.size(g);
            std::printf("%d:", g);
            if (full) {
                for (int j = 0; j < n; ++j) std::printf(" %d", wg.tile(g, j));
            } else {
                std::printf(" %d %d %d", n, n > 0 ? wg.tile(g, 0) : -1, n > 0 ? wg.tile(g, n - 1) : -1);
            }
            std::printf("\n");
        }
        std::printf("end\n");
    }
    return 0;
}
