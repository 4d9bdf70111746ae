// policy_probe.cc -- prints the library's automatic host-side choices for the
// problems given on the command line, compiled with a plain C++ compiler
// against the library's own policy header (tests/test_policy.py drives it).
//
//   split  T slots sm_count nkt mode      -> "dp_tiles splits kt_slice"
//   transpose other M N K mode            -> "0" or "1"
//   panel  M N K f32 ctas_per_sm cta_group multicast sm_count -> "rows"
//   tcshape M N cta_group tile_n multicast sm_count         -> "cta_group tile_n"
//   tcsplit T slots tile_n cta_group multicast mode          -> "split_from"
//   sk T slots sm_count nkt mode                               -> "dp_tiles sk_ctas"
//   kpieces panels out_bytes K                    -> "pieces bound_0 .. bound_pieces"
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "policy.h"

static long long arg(char** argv, int i) { return std::atoll(argv[i]); }

int main(int argc, char** argv) {
    using namespace libgemm;
    if (argc >= 7 && std::strcmp(argv[1], "split") == 0) {
        const TailSplit t = plan_tail_split(arg(argv, 2), (int)arg(argv, 3), (int)arg(argv, 4),
                                            (int)arg(argv, 5), (int)arg(argv, 6));
        std::printf("%d %d %d\n", t.dp_tiles, t.splits, t.kt_slice);
        return 0;
    }
    if (argc >= 7 && std::strcmp(argv[1], "transpose") == 0) {
        std::printf("%d\n", want_transpose(arg(argv, 2), arg(argv, 3), arg(argv, 4), arg(argv, 5),
                                           (int)arg(argv, 6)) ? 1 : 0);
        return 0;
    }
    if (argc >= 10 && std::strcmp(argv[1], "panel") == 0) {
        std::printf("%lld\n",
                    (long long)host_panel_rows(arg(argv, 2), arg(argv, 3), arg(argv, 4),
                                               arg(argv, 5) != 0, (int)arg(argv, 6),
                                               (int)arg(argv, 7), (int)arg(argv, 8),
                                               (int)arg(argv, 9)));
        return 0;
    }
    if (argc >= 8 && std::strcmp(argv[1], "tcshape") == 0) {
        const TcShape t = plan_tc_shape(arg(argv, 2), arg(argv, 3), (int)arg(argv, 4),
                                        (int)arg(argv, 5), arg(argv, 6) != 0, (int)arg(argv, 7));
        std::printf("%d %d\n", t.cta_group, t.tile_n);
        return 0;
    }
    if (argc >= 8 && std::strcmp(argv[1], "tcsplit") == 0) {
        std::printf("%lld\n", (long long)plan_tc_split(arg(argv, 2), arg(argv, 3),
                                                        (int)arg(argv, 4), (int)arg(argv, 5),
                                                        arg(argv, 6) != 0, (int)arg(argv, 7)));
        return 0;
    }
    if (argc >= 7 && std::strcmp(argv[1], "sk") == 0) {
        const StreamK k = plan_stream_k(arg(argv, 2), (int)arg(argv, 3), (int)arg(argv, 4),
                                        (int)arg(argv, 5), (int)arg(argv, 6));
        std::printf("%d %d\n", k.dp_tiles, k.sk_ctas);
        return 0;
    }
    if (argc >= 5 && std::strcmp(argv[1], "kpieces") == 0) {
        const int n = host_k_pieces(arg(argv, 2), (int)arg(argv, 3), arg(argv, 4));
        std::printf("%d", n);
        for (int j = 0; j <= n; ++j)
            std::printf(" %lld", (long long)host_k_bound(arg(argv, 4), n, j));
        std::printf("\n");
        return 0;
    }
    std::fprintf(stderr, "usage: see the header of policy_probe.cc\n");
    return 2;
}
