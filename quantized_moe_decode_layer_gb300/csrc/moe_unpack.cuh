// Packed b-bit codes as floats without an integer-to-float conversion.
//
// A code q at bit position p < 23 of a 32-bit word, with every other bit
// masked off, is read as the IEEE-754 single q * 2^(p - 149) (a subnormal for
// the positions used here, exact).  The decode kernel multiplies it by the
// activation stored times 2^100, which gives q * x * 2^(p - 49) as an exact
// fp32 product, and scales each per-position ("class") sum back by
// 2^(49 - p); or it first multiplies the masked code by 2^(126 - p) to get
// q * 2^-23.  Either way one bitwise AND (a LOP3) per code is the only
// integer work, plus one shift for every few codes that sit above bit 22.
// (The idea of building floats from code bits is the one behind the
// "magic number" conversions of quantised GEMM kernels, e.g. Kim et al.
// 2022, "Who Says Elephants Can't Run".)
//
// A 16-code sub-group of the canonical LSB-first stream (BITS/2 words) is
// read as 8 pairs: pair i = codes (2i, 2i+1), at positions (pa(i), pb(i)),
// accumulated in class cls(i).
#pragma once

#include <cstdint>

namespace moe {

__host__ __device__ __forceinline__ float u2f(uint32_t u)
{
#ifdef __CUDA_ARCH__
    return __uint_as_float(u);
#else
    float f;
    __builtin_memcpy(&f, &u, 4);
    return f;
#endif
}

__host__ __device__ __forceinline__ uint32_t funnel_r(uint32_t lo, uint32_t hi, int s)
{
#ifdef __CUDA_ARCH__
    return __funnelshift_r(lo, hi, s);
#else
    return (uint32_t)((((uint64_t)hi << 32) | lo) >> s);
#endif
}

__host__ __device__ __forceinline__ float mk(uint32_t v, uint32_t m) { return u2f(v & m); }

// 2^(49 - p): brings a class sum of (masked code) * (x * 2^100) back to q x.
__host__ __device__ constexpr uint32_t cls_bits(int p) { return (uint32_t)(49 - p + 127) << 23; }
// 2^(126 - p): turns a masked code into q * 2^-23.
__host__ __device__ constexpr uint32_t fm_bits(int p) { return (uint32_t)(126 - p + 127) << 23; }

struct Pair2 { float a, b; };

template <int BITS> struct Pairs;

template <> struct Pairs<6> {
    // code c at stream bits [6c, 6c + 6); codes 3, 4, 9, 14, 15 are read
    // after a 12-bit shift of their word, codes 5 and 10 (which straddle two
    // words) after a funnel shift
    static constexpr int NC = 7;
    __host__ __device__ static constexpr int pa(int i)
    {
        return i == 0 ? 0 : i == 1 ? 12 : i == 2 ? 12 : i == 3 ? 4 : i == 4 ? 16 : i == 5 ? 0 : 8;
    }
    __host__ __device__ static constexpr int pb(int i)
    {
        return i == 0 ? 6 : i == 1 ? 6 : i == 2 ? 0 : i == 3 ? 10 : i == 4 ? 10 : i == 5 ? 2 : 14;
    }
    __host__ __device__ static constexpr int cls(int i) { return i < 7 ? i : 6; }
    template <typename F>
    __host__ __device__ __forceinline__ static void each(const uint32_t *w, F &&f)
    {
        const uint32_t s0 = w[0] >> 12, s1 = w[1] >> 12, s2 = w[2] >> 12;
        const uint32_t f5 = funnel_r(w[0], w[1], 30), f10 = funnel_r(w[1], w[2], 28);
        constexpr uint32_t M = 0x3Fu;
        f(0, mk(w[0], M), mk(w[0], M << 6));
        f(1, mk(w[0], M << 12), mk(s0, M << 6));
        f(2, mk(s0, M << 12), mk(f5, M));
        f(3, mk(w[1], M << 4), mk(w[1], M << 10));
        f(4, mk(w[1], M << 16), mk(s1, M << 10));
        f(5, mk(f10, M), mk(w[2], M << 2));
        f(6, mk(w[2], M << 8), mk(w[2], M << 14));
        f(7, mk(s2, M << 8), mk(s2, M << 14));
    }
    template <typename P2>
    __host__ __device__ __forceinline__ static void get(const uint32_t *w, P2 (&p)[8])
    {
        const uint32_t s0 = w[0] >> 12, s1 = w[1] >> 12, s2 = w[2] >> 12;
        const uint32_t f5 = funnel_r(w[0], w[1], 30), f10 = funnel_r(w[1], w[2], 28);
        constexpr uint32_t M = 0x3Fu;
        p[0] = {mk(w[0], M), mk(w[0], M << 6)};
        p[1] = {mk(w[0], M << 12), mk(s0, M << 6)};
        p[2] = {mk(s0, M << 12), mk(f5, M)};
        p[3] = {mk(w[1], M << 4), mk(w[1], M << 10)};
        p[4] = {mk(w[1], M << 16), mk(s1, M << 10)};
        p[5] = {mk(f10, M), mk(w[2], M << 2)};
        p[6] = {mk(w[2], M << 8), mk(w[2], M << 14)};
        p[7] = {mk(s2, M << 8), mk(s2, M << 14)};
    }
};

template <> struct Pairs<8> {
    // word j: codes 4j .. 4j+3, one per byte; the high half shifted down
    static constexpr int NC = 1;
    __host__ __device__ static constexpr int pa(int) { return 0; }
    __host__ __device__ static constexpr int pb(int) { return 8; }
    __host__ __device__ static constexpr int cls(int) { return 0; }
    template <typename F>
    __host__ __device__ __forceinline__ static void each(const uint32_t *w, F &&f)
    {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = w[j], s = v >> 16;
            f(2 * j, mk(v, 0xFFu), mk(v, 0xFF00u));
            f(2 * j + 1, mk(s, 0xFFu), mk(s, 0xFF00u));
        }
    }
    template <typename P2>
    __host__ __device__ __forceinline__ static void get(const uint32_t *w, P2 (&p)[8])
    {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t v = w[j], s = v >> 16;
            p[2 * j] = {mk(v, 0xFFu), mk(v, 0xFF00u)};
            p[2 * j + 1] = {mk(s, 0xFFu), mk(s, 0xFF00u)};
        }
    }
};

template <> struct Pairs<4> {
    // word j: codes 8j .. 8j+7, low nibble first; the high half shifted down
    static constexpr int NC = 2;
    __host__ __device__ static constexpr int pa(int i) { return (i & 1) ? 8 : 0; }
    __host__ __device__ static constexpr int pb(int i) { return (i & 1) ? 12 : 4; }
    __host__ __device__ static constexpr int cls(int i) { return i & 1; }
    template <typename F>
    __host__ __device__ __forceinline__ static void each(const uint32_t *w, F &&f)
    {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t v = w[j], s = v >> 16;
            f(4 * j, mk(v, 0xFu), mk(v, 0xF0u));
            f(4 * j + 1, mk(v, 0xF00u), mk(v, 0xF000u));
            f(4 * j + 2, mk(s, 0xFu), mk(s, 0xF0u));
            f(4 * j + 3, mk(s, 0xF00u), mk(s, 0xF000u));
        }
    }
    template <typename P2>
    __host__ __device__ __forceinline__ static void get(const uint32_t *w, P2 (&p)[8])
    {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t v = w[j], s = v >> 16;
            p[4 * j] = {mk(v, 0xFu), mk(v, 0xF0u)};
            p[4 * j + 1] = {mk(v, 0xF00u), mk(v, 0xF000u)};
            p[4 * j + 2] = {mk(s, 0xFu), mk(s, 0xF0u)};
            p[4 * j + 3] = {mk(s, 0xF00u), mk(s, 0xF000u)};
        }
    }
};

// Host check of the tables above against a plain bit-by-bit extraction of
// the stream: every masked code times 2^(149 - p) must be the code, the
// class of a pair must fix both positions, and the scale constants must be
// the powers of two they stand for.  Returns the number of mismatches.
template <int BITS>
inline int pairs_selftest_one(const uint32_t *w)
{
    using PT = Pairs<BITS>;
    int bad = 0;
    Pair2 p[8];
    PT::get(w, p);
    for (int c = 0; c < 16; ++c) {
        uint32_t v = 0;
        for (int t = 0; t < BITS; ++t) {
            const int pos = c * BITS + t;
            v |= ((w[pos >> 5] >> (pos & 31)) & 1u) << t;
        }
        const int i = c / 2;
        const int pos = (c & 1) ? PT::pb(i) : PT::pa(i);
        const float m = (c & 1) ? p[i].b : p[i].a;
        // exact: multiply by 2^(149 - pos) in two power-of-two steps
        const double q = (double)m * 0x1p100 * (double)(1ull << (49 - pos));
        if (q != (double)v) ++bad;
        if ((double)u2f(fm_bits(pos)) * (double)m != (double)v * 0x1p-23) ++bad;
    }
    for (int i = 0; i < 8; ++i)
        for (int j = 0; j < 8; ++j)
            if (PT::cls(i) == PT::cls(j) && (PT::pa(i) != PT::pa(j) || PT::pb(i) != PT::pb(j))) ++bad;
    for (int pos = 0; pos < 23; ++pos)
        if ((double)u2f(cls_bits(pos)) != (double)(1ull << (49 - pos))) ++bad;
    return bad;
}

inline int unpack_selftest_host()
{
    int bad = 0;
    uint32_t seed = 12345u;
    for (int rep = 0; rep < 2000; ++rep) {
        uint32_t w[4];
        for (int i = 0; i < 4; ++i) { seed = seed * 1664525u + 1013904223u; w[i] = seed ^ (seed >> 13); }
        bad += pairs_selftest_one<4>(w);
        bad += pairs_selftest_one<6>(w);
        bad += pairs_selftest_one<8>(w);
    }
    return bad;
}

}  // namespace moe
