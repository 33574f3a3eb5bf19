// Host check of fast_div / fast_div_apply (ssu_device.cuh), the multiply-shift division the
// multi-token kernel uses to turn a tile number into (request, head, slab): for every divisor
// d in 1..70000 and for d at every power of two and its neighbours up to 2^31 - 1, at the
// numerators where a wrong floor would first show (k d - 1, k d, k d + d - 1 for the first
// and last multiples below 2^31, and for every multiple up to 2^20), and at 0 and 2^31 - 1,
// fast_div_apply(n, fast_div(d)) == n / d; then 4 million random pairs.  Prints "ok" or the first counterexample.
#include <cstdio>

#include "ssu_device.cuh"

static long long checked = 0;

static bool check(unsigned long long n, unsigned d, FastDiv f) {
    if (n >= (1ull << 31)) return true;
    ++checked;
    if (fast_div_apply(static_cast<unsigned>(n), f) != n / d) {
        printf("FAIL n %llu d %u: %u != %llu\n", n, d, fast_div_apply(static_cast<unsigned>(n), f),
               n / d);
        return false;
    }
    return true;
}

static bool check_divisor(unsigned d) {
    const FastDiv f = fast_div(d);
    const unsigned long long top = (1ull << 31) - 1;
    if (!check(0, d, f) || !check(top, d, f)) return false;
    const unsigned long long kmax = top / d;
    for (unsigned long long k = 1; k <= kmax; ++k) {
        const unsigned long long n = k * d;
        if (!check(n - 1, d, f) || !check(n, d, f) || !check(n + d - 1, d, f)) return false;
        if (n > (1ull << 20) && k + 4 < kmax) k = kmax - 4;  // then the last few multiples
    }
    return true;
}

int main() {
    for (unsigned d = 1; d <= 70000; ++d)
        if (!check_divisor(d)) return 1;
    for (unsigned e = 17; e < 31; ++e)
        for (long long delta = -2; delta <= 2; ++delta)
            if (!check_divisor(static_cast<unsigned>((1ll << e) + delta))) return 1;
    if (!check_divisor(2147483647u)) return 1;
    // 4 million random (n, d) pairs from a 64-bit linear congruential generator.
    unsigned long long x = 0x9E3779B97F4A7C15ull;
    for (int i = 0; i < 4000000; ++i) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        const unsigned n = static_cast<unsigned>(x >> 33);
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        unsigned d = static_cast<unsigned>(x >> (33 + (x & 31) % 31));
        if (d == 0) d = 1;
        if (!check(n, d, fast_div(d))) return 1;
    }
    printf("ok\n");
    fprintf(stderr, "%lld cases\n", checked);
    return 0;
}
