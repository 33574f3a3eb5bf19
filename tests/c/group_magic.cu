// Host check of group_of / group_magic (ssu_device.cuh), the division-free group index: for
// every divisor d in 1..65535 and every head index at and around each multiple of d below
// 2^16 (where a wrong floor would first show), group_of(h, group_magic(d)) == h / d.
// Prints "ok" or the first counterexample.
#include <cstdio>

#include "ssu_device.cuh"

int main() {
    long long checked = 0;
    for (unsigned d = 1; d < 65536; ++d) {
        const unsigned long long m = group_magic(d);
        for (unsigned k = 0; k * d < 65536; ++k) {
            const long long cand[3] = {static_cast<long long>(k) * d - 1,
                                       static_cast<long long>(k) * d,
                                       static_cast<long long>(k) * d + d - 1};
            for (long long h : cand) {
                if (h < 0 || h > 65535) continue;
                ++checked;
                if (group_of(static_cast<int>(h), m) != static_cast<int>(h / d)) {
                    printf("FAIL h %lld d %u: %d != %lld\n", h, d,
                           group_of(static_cast<int>(h), m), h / d);
                    return 1;
                }
            }
        }
    }
    printf("ok\n");
    fprintf(stderr, "%lld cases\n", checked);
    return 0;
}
