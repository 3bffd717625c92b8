// Host-only check of santa::point_fraction against IEEE double arithmetic: for every S in
// 1..4096 (rS = the double nearest 1/S), random points s < S and random Philox words
// (plus the words of u = 0, u = 1 - 2^-32 and small u), floor(((s + u) * rS) * 2^64) in
// doubles must equal the integer evaluation.  Prints the count; exits 1 on a mismatch.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>

#include "../../stochastic_sparse_kv_gb300/csrc/santa_common.cuh"

int main()
{
    std::mt19937_64 rng(20261202);
    long long n = 0, bad = 0;
    for (int S = 1; S <= 4096; ++S) {
        const double rS = 1.0 / (double)S;
        uint64_t rb;
        std::memcpy(&rb, &rS, 8);
        const int trials = (S <= 64 || (S & (S - 1)) == 0) ? 4000 : 300;
        for (int t = 0; t < trials; ++t) {
            const int s = (t < 16) ? (t & 1 ? S - 1 : 0) : (int)(rng() % (uint64_t)S);
            uint64_t w = rng();
            if (t < 8) w = (t & 2) ? ~0ull : 0ull;
            else if (t < 16) w = (uint64_t)(t - 8) << 32;
            const double u = (double)(uint32_t)(w >> 32) * 0x1p-32;
            const double tt = ((double)s + u) * rS;
            const uint64_t want = (uint64_t)(tt * 0x1p64);
            const uint64_t got = santa::point_fraction(s, w, rb);
            ++n;
            if (got != want) {
                if (bad < 10)
                    std::printf("S=%d s=%d word=%016llx: double %016llx, integer %016llx\n", S, s,
                                (unsigned long long)w, (unsigned long long)want, (unsigned long long)got);
                ++bad;
            }
        }
    }
    std::printf("%lld points, %lld mismatches\n", n, bad);
    return bad != 0;
}
