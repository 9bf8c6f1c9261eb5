// Exact conversion of packed b-bit codes to fp32, 16 codes (one sub-group)
// at a time, from the LSB-first bit stream of the device layout.
//
// Method: IEEE-754 bit construction (the same idea as the "magic number"
// int-to-float conversions used for quantised GEMMs, e.g. Kim et al. 2022,
// "Who Says Elephants Can't Run"): for a code q sitting at bit position p of
// a 32-bit word, OR-ing the word (masked to the code) with the exponent field
// (150 - p) << 23 gives the float 2^(23-p) + q exactly, because q << p then
// lies inside the 23-bit mantissa with unit weight 2^(23-p-23+p) = 1.
// Subtracting the constant 2^(23-p) returns q exactly.  Choosing the exponent
// per bit position avoids shifting each code down to bit 0: one LOP3-style
// AND/OR plus one FADD per code, plus one shift per few codes.
#pragma once

#include <cstdint>
#include <initializer_list>

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

// Code of `BITS` bits at position P of v, as an exact float.
template <int BITS, int P>
__host__ __device__ __forceinline__ float code_at(uint32_t v)
{
    static_assert(P + BITS <= 23, "code must sit inside the mantissa");
    constexpr uint32_t kMask = ((1u << BITS) - 1u) << P;
    constexpr uint32_t kExp = (uint32_t)(150 - P) << 23;
    return u2f((v & kMask) | kExp) - u2f(kExp);
}

// Raw form: the float 2^(23-P) + q (no subtraction yet) and its offset
// 2^(23-P); packed two-lane FADD then removes the offsets of a pair at once.
template <int BITS, int P>
__host__ __device__ __forceinline__ float code_raw(uint32_t v)
{
    static_assert(P + BITS <= 23, "code must sit inside the mantissa");
    constexpr uint32_t kMask = ((1u << BITS) - 1u) << P;
    constexpr uint32_t kExp = (uint32_t)(150 - P) << 23;
    return u2f((v & kMask) | kExp);
}

template <int P>
__host__ __device__ __forceinline__ float code_off()
{
    return u2f((uint32_t)(150 - P) << 23);
}

// Codes 4t .. 4t+3 of a 16-code sub-group held in w[] (BITS/2 words).
// get4 gives exact floats; raw4 gives code_raw values f and offsets o with
// f - o the codes.
template <int BITS>
struct Unpack;

template <>
struct Unpack<4> {
    // word i holds codes 8i .. 8i+7 at bits 0, 4, ..., 28
    template <int T>
    __host__ __device__ __forceinline__ static void get4(const uint32_t *w, float *q)
    {
        const uint32_t v = w[T >> 1];
        if ((T & 1) == 0) {
            q[0] = code_at<4, 0>(v);
            q[1] = code_at<4, 4>(v);
            q[2] = code_at<4, 8>(v);
            q[3] = code_at<4, 12>(v);
        } else {
            const uint32_t s = v >> 12;   // codes 5, 6, 7 of the word move to 8, 12, 16
            q[0] = code_at<4, 16>(v);
            q[1] = code_at<4, 8>(s);
            q[2] = code_at<4, 12>(s);
            q[3] = code_at<4, 16>(s);
        }
    }
    template <int T>
    __host__ __device__ __forceinline__ static void raw4(const uint32_t *w, float *f, float *o)
    {
        const uint32_t v = w[T >> 1];
        if ((T & 1) == 0) {
            f[0] = code_raw<4, 0>(v); o[0] = code_off<0>();
            f[1] = code_raw<4, 4>(v); o[1] = code_off<4>();
            f[2] = code_raw<4, 8>(v); o[2] = code_off<8>();
            f[3] = code_raw<4, 12>(v); o[3] = code_off<12>();
        } else {
            const uint32_t s = v >> 12;
            f[0] = code_raw<4, 16>(v); o[0] = code_off<16>();
            f[1] = code_raw<4, 8>(s); o[1] = code_off<8>();
            f[2] = code_raw<4, 12>(s); o[2] = code_off<12>();
            f[3] = code_raw<4, 16>(s); o[3] = code_off<16>();
        }
    }
};

template <>
struct Unpack<8> {
    // word i holds codes 4i .. 4i+3, one per byte
    template <int T>
    __host__ __device__ __forceinline__ static void get4(const uint32_t *w, float *q)
    {
        const uint32_t v = w[T];
        const uint32_t s = v >> 16;
        q[0] = code_at<8, 0>(v);
        q[1] = code_at<8, 8>(v);
        q[2] = code_at<8, 0>(s);
        q[3] = code_at<8, 8>(s);
    }
    template <int T>
    __host__ __device__ __forceinline__ static void raw4(const uint32_t *w, float *f, float *o)
    {
        const uint32_t v = w[T];
        const uint32_t s = v >> 16;
        f[0] = code_raw<8, 0>(v); o[0] = code_off<0>();
        f[1] = code_raw<8, 8>(v); o[1] = code_off<8>();
        f[2] = code_raw<8, 0>(s); o[2] = code_off<0>();
        f[3] = code_raw<8, 8>(s); o[3] = code_off<8>();
    }
};

template <>
struct Unpack<6> {
    // 16 codes in 96 bits: code i at stream bits 6i .. 6i+5.  Word 0 holds
    // codes 0-4 and the low 2 bits of code 5; word 1 the high 4 bits of
    // code 5, codes 6-9 and the low 4 bits of code 10; word 2 the high 2 bits
    // of code 10 and codes 11-15.
    template <int T>
    __host__ __device__ __forceinline__ static void get4(const uint32_t *w, float *q)
    {
        if (T == 0) {          // codes 0..3
            const uint32_t s0 = w[0] >> 12;
            q[0] = code_at<6, 0>(w[0]);
            q[1] = code_at<6, 6>(w[0]);
            q[2] = code_at<6, 12>(w[0]);
            q[3] = code_at<6, 6>(s0);
        } else if (T == 1) {   // codes 4..7
            const uint32_t s0 = w[0] >> 12;
            q[0] = code_at<6, 12>(s0);
            q[1] = code_at<6, 0>(funnel_r(w[0], w[1], 30));
            q[2] = code_at<6, 4>(w[1]);
            q[3] = code_at<6, 10>(w[1]);
        } else if (T == 2) {   // codes 8..11
            const uint32_t s1 = w[1] >> 12;
            q[0] = code_at<6, 16>(w[1]);
            q[1] = code_at<6, 10>(s1);
            q[2] = code_at<6, 0>(funnel_r(w[1], w[2], 28));
            q[3] = code_at<6, 2>(w[2]);
        } else {               // codes 12..15
            const uint32_t s2 = w[2] >> 12;
            q[0] = code_at<6, 8>(w[2]);
            q[1] = code_at<6, 14>(w[2]);
            q[2] = code_at<6, 8>(s2);
            q[3] = code_at<6, 14>(s2);
        }
    }
    template <int T>
    __host__ __device__ __forceinline__ static void raw4(const uint32_t *w, float *f, float *o)
    {
        if (T == 0) {
            const uint32_t s0 = w[0] >> 12;
            f[0] = code_raw<6, 0>(w[0]); o[0] = code_off<0>();
            f[1] = code_raw<6, 6>(w[0]); o[1] = code_off<6>();
            f[2] = code_raw<6, 12>(w[0]); o[2] = code_off<12>();
            f[3] = code_raw<6, 6>(s0); o[3] = code_off<6>();
        } else if (T == 1) {
            const uint32_t s0 = w[0] >> 12;
            f[0] = code_raw<6, 12>(s0); o[0] = code_off<12>();
            f[1] = code_raw<6, 0>(funnel_r(w[0], w[1], 30)); o[1] = code_off<0>();
            f[2] = code_raw<6, 4>(w[1]); o[2] = code_off<4>();
            f[3] = code_raw<6, 10>(w[1]); o[3] = code_off<10>();
        } else if (T == 2) {
            const uint32_t s1 = w[1] >> 12;
            f[0] = code_raw<6, 16>(w[1]); o[0] = code_off<16>();
            f[1] = code_raw<6, 10>(s1); o[1] = code_off<10>();
            f[2] = code_raw<6, 0>(funnel_r(w[1], w[2], 28)); o[2] = code_off<0>();
            f[3] = code_raw<6, 2>(w[2]); o[3] = code_off<2>();
        } else {
            const uint32_t s2 = w[2] >> 12;
            f[0] = code_raw<6, 8>(w[2]); o[0] = code_off<8>();
            f[1] = code_raw<6, 14>(w[2]); o[1] = code_off<14>();
            f[2] = code_raw<6, 8>(s2); o[2] = code_off<8>();
            f[3] = code_raw<6, 14>(s2); o[3] = code_off<14>();
        }
    }
};

// Host check of the tables above against a plain bit-by-bit extraction.
// Returns the number of mismatching codes over a fixed pseudo-random set.
inline int unpack_selftest_host()
{
    int bad = 0;
    uint32_t seed = 12345u;
    for (int rep = 0; rep < 2000; ++rep) {
        uint32_t w[4];
        for (int i = 0; i < 4; ++i) { seed = seed * 1664525u + 1013904223u; w[i] = seed ^ (seed >> 13); }
        for (int bits : {4, 6, 8}) {
            float q[16];
            if (bits == 4) {
                Unpack<4>::get4<0>(w, q); Unpack<4>::get4<1>(w, q + 4); Unpack<4>::get4<2>(w, q + 8); Unpack<4>::get4<3>(w, q + 12);
            } else if (bits == 6) {
                Unpack<6>::get4<0>(w, q); Unpack<6>::get4<1>(w, q + 4); Unpack<6>::get4<2>(w, q + 8); Unpack<6>::get4<3>(w, q + 12);
            } else {
                Unpack<8>::get4<0>(w, q); Unpack<8>::get4<1>(w, q + 4); Unpack<8>::get4<2>(w, q + 8); Unpack<8>::get4<3>(w, q + 12);
            }
            float fr[16], of[16];
            if (bits == 4) {
                Unpack<4>::raw4<0>(w, fr, of); Unpack<4>::raw4<1>(w, fr + 4, of + 4); Unpack<4>::raw4<2>(w, fr + 8, of + 8); Unpack<4>::raw4<3>(w, fr + 12, of + 12);
            } else if (bits == 6) {
                Unpack<6>::raw4<0>(w, fr, of); Unpack<6>::raw4<1>(w, fr + 4, of + 4); Unpack<6>::raw4<2>(w, fr + 8, of + 8); Unpack<6>::raw4<3>(w, fr + 12, of + 12);
            } else {
                Unpack<8>::raw4<0>(w, fr, of); Unpack<8>::raw4<1>(w, fr + 4, of + 4); Unpack<8>::raw4<2>(w, fr + 8, of + 8); Unpack<8>::raw4<3>(w, fr + 12, of + 12);
            }
            for (int i = 0; i < 16; ++i) {
                if (fr[i] - of[i] != q[i]) ++bad;
                uint32_t v = 0;
                for (int t = 0; t < bits; ++t) {
                    const int pos = i * bits + t;
                    v |= ((w[pos >> 5] >> (pos & 31)) & 1u) << t;
                }
                if (q[i] != (float)v) ++bad;
            }
        }
    }
    return bad;
}

}  // namespace moe
