// Host-side harness for the work-queue builders the fused kernel's schedule
// comes from: build_queues (the host path) and, with the argument
// "parallel", the plan kernel's parallel form (queue_counts, queue1_part,
// queue2_part) run one position after another with the prefix sums the
// kernel takes between its steps.  Reads cases from stdin, one per line:
//   E n_slabs n_slabs2 two_pass ready_first lookahead M_0 ... M_{E-1}
// (n_slabs: slabs per band of the amax / single-pass items, n_slabs2: of the
// encode items)
// orders the non-empty experts as the host path does (by decreasing size,
// stable, for the two-pass recipe; by index otherwise), builds the queues and
// prints, per case, "n_items n_segs1 n_items2 n_segs" and then one line
// "start kind expert first" per segment.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "gsa_kernel.cuh"

using namespace gsa;

// The plan kernel's queue build, thread by thread.
void build_parallel(PlanTab &T, const int *order, int n, int n_slabs, int n_slabs2, bool two_pass, bool ready_first,
                    int lookahead) {
    static QueueScan Q;
    std::vector<int> a(n + 1), b(n + 1);
    for (int t = 0; t <= n; ++t) queue_counts(T, order, n, n_slabs, n_slabs2, t, a[t], b[t]);
    Q.c[0] = Q.c2[0] = 0;
    for (int t = 0; t < n; ++t) {
        Q.c[t + 1] = Q.c[t] + a[t];
        Q.c2[t + 1] = Q.c2[t] + b[t];
    }
    for (int t = 0; t <= n; ++t) queue1_part<false>(T, Q, order, n, two_pass, ready_first, lookahead, t, a[t], b[t]);
    int segs = 0, items = 0;
    for (int t = 0; t <= n; ++t) {
        Q.so[t] = segs;
        Q.io[t] = items;
        segs += a[t];
        items += b[t];
    }
    for (int t = 0; t <= n; ++t) {
        queue1_part<true>(T, Q, order, n, two_pass, ready_first, lookahead, t, a[t], b[t]);
        queue2_part(T, Q, order, n, two_pass, ready_first, items, segs, t);
    }
}

int main(int argc, char **argv) {
    const bool parallel = argc > 1 && std::strcmp(argv[1], "parallel") == 0;
    int E, n_slabs, n_slabs2, two_pass, ready_first, lookahead;
    static PlanTab T;
    while (std::scanf("%d %d %d %d %d %d", &E, &n_slabs, &n_slabs2, &two_pass, &ready_first, &lookahead) == 6) {
        std::vector<long long> m(E);
        for (int e = 0; e < E; ++e)
            if (std::scanf("%lld", &m[e]) != 1) return 1;
        T.band_start[0] = 0;
        for (int e = 0; e < E; ++e) T.band_start[e + 1] = T.band_start[e] + static_cast<int>((m[e] + kRows - 1) / kRows);
        std::vector<int> order;
        for (int e = 0; e < E; ++e)
            if (m[e] > 0) order.push_back(e);
        if (two_pass) std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return m[a] > m[b]; });
        std::vector<int> pe(order.size() + 1), pp(order.size() + 1);
        if (parallel)
            build_parallel(T, order.data(), static_cast<int>(order.size()), n_slabs, n_slabs2, two_pass != 0,
                           ready_first != 0, lookahead);
        else
            build_queues(T, order.data(), static_cast<int>(order.size()), n_slabs, n_slabs2, two_pass != 0,
                         ready_first != 0, lookahead, pe.data(), pp.data());
        std::printf("%d %d %d %d\n", T.n_items, T.n_segs1, T.n_items2, T.n_segs);
        for (int i = 0; i < T.n_segs; ++i)
            std::printf("%d %d %d %d\n", T.seg_start[i], T.seg_info[i] >> 16, T.seg_info[i] & 0xFFFF, T.seg_first[i]);
    }
    return 0;
}
