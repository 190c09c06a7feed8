// Host-side check of the launch-time divider of kda_prep_impl.cuh (FastDiv):
// floor(n / d) for every divisor 1 .. 4096 and a spread of larger ones, at
// the numerators where a multiply-high division would first go wrong (each
// multiple of d and its neighbours, and the top of the 31-bit range).
// Built and run by tests/test_abi_host.py; prints "ok" and exits 0 when every
// quotient matches.
#include <cstdio>
#include <cstdlib>

#include "kda_prep_impl.cuh"

static int check(uint32_t d, uint32_t n) {
    const kda::prep::FastDiv f = kda::prep::make_fastdiv(d);
    if (kda::prep::fast_div(n, f) != n / d) {
        std::printf("d=%u n=%u got %u want %u\n", d, n, kda::prep::fast_div(n, f), n / d);
        return 1;
    }
    return 0;
}

int main() {
    const uint32_t top = 0x7fffffffu;
    int bad = 0;
    uint64_t state = 0x9e3779b97f4a7c15ull;
    auto next = [&state]() {   // splitmix64
        uint64_t z = (state += 0x9e3779b97f4a7c15ull);
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        return z ^ (z >> 31);
    };
    for (uint32_t d = 1; d <= 4096 && bad < 10; ++d) {
        for (uint32_t n = 0; n < 4 * d + 3; ++n) bad += check(d, n);
        for (int i = 0; i < 2000; ++i) {
            const uint32_t q = static_cast<uint32_t>(next() % (top / d + 1));
            const uint64_t base = static_cast<uint64_t>(q) * d;
            for (int delta = -1; delta <= 1; ++delta) {
                const int64_t n = static_cast<int64_t>(base) + delta;
                if (n >= 0 && n <= top) bad += check(d, static_cast<uint32_t>(n));
            }
        }
        for (uint32_t n = top - 3 * d; n <= top - d + 1 && n <= top; n += d) bad += check(d, n);
        bad += check(d, top);
    }
    for (int i = 0; i < 20000 && bad < 10; ++i) {
        const uint32_t d = 1 + static_cast<uint32_t>(next() % top);
        const uint32_t q = static_cast<uint32_t>(next() % (top / d + 1));
        const uint64_t base = static_cast<uint64_t>(q) * d;
        for (int delta = -1; delta <= 1; ++delta) {
            const int64_t n = static_cast<int64_t>(base) + delta;
            if (n >= 0 && n <= top) bad += check(d, static_cast<uint32_t>(n));
        }
        bad += check(d, top);
        bad += check(d, static_cast<uint32_t>(next() % (uint64_t(top) + 1)));
    }
    for (uint32_t k = 0; k < 31; ++k)   // powers of two and their neighbours
        for (uint32_t d : {(1u << k) - 1, 1u << k, (1u << k) + 1})
            if (d >= 1 && d <= top) {
                bad += check(d, top);
                bad += check(d, top - 1);
                bad += check(d, d);
                bad += check(d, d - 1);
            }
    if (bad) return 1;
    std::printf("ok\n");
    return 0;
}
