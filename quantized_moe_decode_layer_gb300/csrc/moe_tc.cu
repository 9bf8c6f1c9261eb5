// Grouped products of the routed experts on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory): the grouped-GEMM regime that
// appears when many token rows share an expert.  Grouped mode (moe_grouped.cu)
// runs a layer's expert products here when a call has more rows than one
// persistent launch holds; up to that the persistent kernel keeps every step
// on the FMA pipes, where each token row's result is bitwise the one-row
// result.
//
// What they compute (an expert FFN as the pages state it: dequantised weight
// w = q * s + b per group of 64 along the input axis, SwiGLU between the two
// projections): for each listed expert e and each token row m in its mask,
//   gate/up:  act[u][m][j] = silu(W_gate,e[j] . hn[m]) * (W_up,e[j] . hn[m])
//   down:     y[u][m][h]   = W_down,e[h] . act[u][m]
// A launch can carry a second set of products (the shared expert, with its
// own weights and code width) beside the first.
//
// Layout and arithmetic:
//   - One CTA per (expert, tile of 128 consecutive weight rows; for gate/up
//     64 units of gate and up rows).  The tile is the MMA's M = 128 dimension.
//   - The token rows are the N dimension: N = 64 = 32 rows of the high fp16
//     halves of the inputs (x with its 13 low mantissa bits cleared: exact in
//     fp16), then 32 rows of the low halves (x - high, rounded to fp16), so
//     the inputs keep ~22 significant bits.  The weights are split the same
//     way (w = fma(q, s, b) in fp32, then the two halves, each an MMA into
//     the same accumulator), so every product term keeps ~21 bits.  Only the
//     final packing of two halves into one f16x2 word is a conversion.
//     (bf16 halves keep only ~16: with outputs that are small differences of
//     terms in the thousands, as the synthetic 6-bit layers give, that
//     missed the output tolerance.)  fp16 bounds the inputs and weights to
//     |v| < 65504.
//   - K runs over the input axis in chunks of 64 (one quantisation group):
//     each of the CTA's 256 threads dequantises half a group of one tile row
//     into shared memory and writes 16 inputs of the token-row chunk next to
//     it, and one thread issues 8 MMAs of K = 16 (high, then low weight
//     halves).  Two register sets of codes, scales and inputs alternate
//     between even and odd chunks; chunk c + 2's loads go out as soon as
//     chunk c has been converted.  Two chunk buffers alternate in shared
//     memory; an MMA batch's commit arrives on the buffer's mbarrier, which
//     the next writers of that buffer wait on.
//   - Shared-memory tiles use the no-swizzle K-major canonical layout: 8x16-
//     byte core matrices of 128 contiguous bytes, 128 B apart along K and
//     1024 B apart along M/N.
//   - Each chunk's MMAs start a fresh fp32 sum in one of four accumulator
//     blocks; two chunks later every warp adds the block into fp32 registers
//     (round to nearest; warps 0-3 the high-half columns, warps 4-7 the low),
//     so the long sum over K is not accumulated inside the tensor core (that
//     drifted beyond the output tolerance on cancelling outputs).
//   - Epilogue: warps 4-7 hand their low-half sums to warps 0-3 (the same
//     tile rows) through shared memory; for gate/up the neighbours 2j, 2j + 1
//     meet through one shuffle for SwiGLU.
// Every wait is bounded; a wait that runs out sets *err and the CTA skips
// the rest of its work, still freeing its tensor memory.

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kTcRows = 128;      // weight rows per tile (MMA M)
constexpr int kTcTok = 32;        // token rows per call at most
constexpr int kTcN = 2 * kTcTok;  // MMA N: high halves, then low halves
constexpr int kTcK = 64;          // input elements per chunk (one group)
constexpr int kTcThreads = 256;
constexpr int kTileA = kTcRows * kTcK * 2;  // bytes of a weight chunk, one fp16 half (16 KB)
constexpr int kTileB = kTcN * kTcK * 2;     // bytes of a token chunk (8 KB)
constexpr int kTcSmem = 4 * kTileA + 2 * kTileB + 64;   // 2 buffers of (A hi, A lo, B)
constexpr uint32_t kTmemCols = 4 * kTcN;    // four fp32 accumulator blocks of N columns

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of element (r, k) of a [rows x 64] fp16 tile in the no-swizzle
// K-major layout (core matrix = 8 rows x 8 elements, 128 contiguous bytes).
__device__ __forceinline__ uint32_t canon(int r, int k)
{
    return (uint32_t)((r >> 3) * 1024 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (between core matrices along K: 128), stride-dimension byte offset
// (between 8-row groups: 1024), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(1024u >> 4) << 32) |
           (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N = kTcN, M = kTcRows.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kTcN >> 3) << 17) |
                            ((uint32_t)(kTcRows >> 4) << 24);

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, unsigned parity, long long timeout_ns)
{
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
#pragma unroll 1
    for (;;) {
        uint32_t done;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (done) return true;
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if ((long long)(t - t0) > timeout_ns) return false;
    }
}

// Two floats as one f16x2 word (a in the low half), one paired conversion.
__device__ __forceinline__ uint32_t pack_h(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The high fp16 half of v without a conversion: v with its 13 low mantissa
// bits cleared has at most 11 significant bits, so it converts to fp16
// exactly (inside fp16's range), and v - hi is exact in fp32.
__device__ __forceinline__ float f16_hi(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

// A code (below 2^23) as a float without a conversion instruction.
__device__ __forceinline__ float code_f(uint32_t q) { return __uint_as_float(q | 0x4B000000u) - 8388608.0f; }

// Code k (0 .. 31) of half a group's LSB-first code stream, held in the
// BITS words w (32 codes of BITS bits).
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[BITS], int k)
{
    const int bit = k * BITS, wi = bit >> 5, off = bit & 31;
    uint32_t v = w[wi] >> off;
    if (off + BITS > 32) v |= w[wi + 1] << (32 - off);
    return v & ((1u << BITS) - 1u);
}

// y[n] += column n (warps 0-3: the high halves) or column 32 + n (warps 4-7:
// the low halves) of accumulator block `blk`; warp w reads tensor-memory
// lanes 32 (w % 4) .. + 31, one tile row per thread.
__device__ __forceinline__ void drain_block(uint32_t taddr, int warp, int blk, float (&y)[kTcTok])
{
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t r[16];
        const uint32_t a = taddr + ((uint32_t)(32 * (warp & 3)) << 16) +
                           (uint32_t)(kTcN * blk + kTcTok * (warp >> 2) + 16 * q);
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                     "%12, %13, %14, %15}, [%16];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                       "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                       "=r"(r[15])
                     : "r"(a)
                     : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int i = 0; i < 16; ++i) y[16 * q + i] += __uint_as_float(r[i]);
    }
}

// One grouped product: for slot u (expert experts[u]) and each token row m
// of masks[u], the expert's `rows` weight rows (K inputs each, row_bytes per
// packed row, rows e * rows .. of W) against input vector
// in[(u * in_u + m) * K ..] (in_u = 0: one vector per row shared by every
// slot; in_u = M: a vector per (slot, row)).  SWIGLU: rows 2j and 2j + 1 are
// gate and up rows, out[(u * M + m) * rows / 2 + j] = silu(gate) * up; else
// out[(u * M + m) * rows + r] = the dot product of row r.
struct TcSet {
    const uint8_t *W;
    int rows, K, row_bytes;
    const float *in;
    int in_u;
    const int32_t *experts;
    const uint32_t *masks;
    const int *U_dev;   // device-side slot count, or NULL
    float *out;
};

template <int BITS, bool SWIGLU>
__device__ __forceinline__ void grouped_tc_body(const TcSet &set, int u, int tile, int M, long long timeout_ns, int *err)
{
    const uint8_t *__restrict__ W = set.W;
    const int rows = set.rows, K = set.K, row_bytes = set.row_bytes, in_u = set.in_u;
    const float *__restrict__ in = set.in;
    const int32_t *__restrict__ experts = set.experts;
    const uint32_t *__restrict__ masks = set.masks;
    float *__restrict__ out = set.out;
    // tiles past this set's rows, and slots at or past a device-side count,
    // have nothing to do
    if (tile * kTcRows >= rows) return;
    if (set.U_dev && u >= *set.U_dev) return;
    extern __shared__ __align__(1024) uint8_t sm[];
    // buffer b: weight halves at A0 + 2 b kTileA (high) and + kTileA (low), tokens at B0 + b kTileB
    uint8_t *const A0 = sm, *const B0 = sm + 4 * kTileA;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + 4 * kTileA + 2 * kTileB);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e = experts[u];
    const uint32_t mask = masks[u];
    const int nr = __popc(mask);

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&bar[1])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *tmem_slot;

    // this thread's half weight row (codes 32 ah .. + 31 of each group of
    // row arow) and its token-chunk share (inputs kq .. + 15 of each chunk of
    // B row brow).  Each warp keeps 16 weight rows and 8 B rows; within every
    // 8 consecutive lanes the row varies and the column does not, so their
    // 16-byte stores fill one 128-byte core-matrix row set with no bank
    // conflict.
    const int arow = ((tid >> 4) << 3) | (tid & 7), ah = (tid >> 3) & 1;
    const uint8_t *row = W + ((size_t)e * rows + (size_t)kTcRows * tile + arow) * (size_t)row_bytes;
    const uint32_t *codes = reinterpret_cast<const uint32_t *>(row) + ah * BITS;   // + c * 2 BITS words
    const uint32_t *sbp = reinterpret_cast<const uint32_t *>(row + (size_t)K * BITS / 8);
    const int brow = ((tid >> 5) << 3) | (tid & 7), kq = ((tid >> 3) & 3) * 16;
    const int tn = brow & (kTcTok - 1);
    const bool lo_half = brow >= kTcTok;
    int trow = tn < nr ? (int)__fns(mask, 0, tn + 1) : -1;
    if (trow >= M) trow = -1;   // mask bits at or above M name no row
    const float4 *hsrc =
        reinterpret_cast<const float4 *>(in + ((size_t)u * in_u + (trow < 0 ? 0 : trow)) * (size_t)K + kq);

    const int G = K / kTcK;
    // Two register sets of loaded codes, scale and inputs alternate between
    // the even and the odd chunks; a set is refilled with chunk c + 2 as soon
    // as chunk c has been converted from it, and is never copied (a copy
    // would wait for the load), so each load has two chunks to land.
    uint32_t wA[BITS], wB[BITS], sbA = 0u, sbB = 0u;
    float4 hA[4], hB[4];
    auto load_set = [&](int c, uint32_t (&w)[BITS], uint32_t &sb, float4 (&h)[4]) {
        if (c < G) {
#pragma unroll
            for (int i = 0; i < BITS; ++i) w[i] = __ldg(codes + c * 2 * BITS + i);
            sb = __ldg(sbp + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (trow >= 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) h[i] = __ldg(hsrc + c * (kTcK / 4) + i);
            }
        }
    };
    load_set(0, wA, sbA, hA);
    load_set(1, wB, sbB, hB);
    bool ok = true;
    // Each chunk's MMAs start a fresh sum in accumulator block c & 3; when
    // chunk c starts, every warp adds chunk c - 2's finished block (warps 0-3
    // its high-half columns, warps 4-7 its low-half columns) into these fp32
    // registers, so the long sums round to nearest here instead of
    // accumulating inside the tensor core over all of K, and the MMAs of
    // chunk c - 1 still run meanwhile.
    float y[kTcTok];
#pragma unroll
    for (int n = 0; n < kTcTok; ++n) y[n] = 0.f;
    auto step = [&](int c, uint32_t (&w0)[BITS], uint32_t &sb0, float4 (&h0)[4]) -> bool {
        const int b = c & 1;
        uint8_t *const Ab = A0 + 2 * b * kTileA, *const Alb = Ab + kTileA, *const Bb = B0 + b * kTileB;
        // the MMAs that last read buffer b (chunk c - 2) must be done (a
        // thread whose wait runs out still takes part in this chunk's
        // barrier, after which the whole CTA stops)
        if (c >= 2) {
            ok = mbar_wait_bounded(su32(&bar[b]), (unsigned)((c - 2) >> 1) & 1u, timeout_ns);
            // the same commit ends chunk c - 2's sums (block (c - 2) & 3)
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (ok) drain_block(taddr, warp, (c - 2) & 3, y);
        }
        // weights: 32 values of row arow, group c, as high and low fp16 halves
        {
            const float sc = __uint_as_float(sb0 << 16), bb = __uint_as_float(sb0 & 0xFFFF0000u);
#pragma unroll
            for (int k8 = 0; k8 < 4; ++k8) {
                uint32_t ph[4], pl[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float wa = fmaf(code_f(code_at<BITS>(w0, 8 * k8 + 2 * j)), sc, bb);
                    const float wb = fmaf(code_f(code_at<BITS>(w0, 8 * k8 + 2 * j + 1)), sc, bb);
                    const float ha = f16_hi(wa), hb = f16_hi(wb);
                    ph[j] = pack_h(ha, hb);
                    pl[j] = pack_h(wa - ha, wb - hb);
                }
                const uint32_t off = canon(arow, 32 * ah + 8 * k8);
                *reinterpret_cast<uint4 *>(Ab + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<uint4 *>(Alb + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
        }
        // token rows: B row brow holds the high (or low) fp16 half of token
        // row trow, inputs 64 c + kq .. + 15
        {
            float v[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[4 * i] = h0[i].x; v[4 * i + 1] = h0[i].y; v[4 * i + 2] = h0[i].z; v[4 * i + 3] = h0[i].w;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float hi = f16_hi(v[i]);
                v[i] = lo_half ? v[i] - hi : hi;
            }
#pragma unroll
            for (int k8 = 0; k8 < 2; ++k8)
                *reinterpret_cast<uint4 *>(Bb + canon(brow, kq + 8 * k8)) =
                    make_uint4(pack_h(v[8 * k8], v[8 * k8 + 1]), pack_h(v[8 * k8 + 2], v[8 * k8 + 3]),
                               pack_h(v[8 * k8 + 4], v[8 * k8 + 5]), pack_h(v[8 * k8 + 6], v[8 * k8 + 7]));
        }
        load_set(c + 2, w0, sb0, h0);
        // the generic-proxy stores above become visible to the tensor core,
        // and the tensor-memory reads above end before the next MMAs
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        ok = __syncthreads_and(ok);
        if (!ok) return false;
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int kk = 0; kk < 2 * (kTcK / 16); ++kk) {
                // high weight halves, then low, into the same accumulator
                const uint8_t *At = kk < kTcK / 16 ? Ab : Alb;
                const int ks = kk % (kTcK / 16);
                const uint64_t ad = smem_desc(su32(At) + ks * 256), bd = smem_desc(su32(Bb) + ks * 256);
                const uint32_t accumulate = kk > 0 ? 1u : 0u;
                asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                             "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(taddr + kTcN * (c & 3)),
                             "l"(ad), "l"(bd), "r"(kIdesc), "r"(accumulate)
                             : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             su32(&bar[b]))
                         : "memory");
        }
        return true;
    };
#pragma unroll 1
    for (int c = 0; c < G; c += 2) {
        if (!step(c, wA, sbA, hA)) break;
        if (c + 1 < G && !step(c + 1, wB, sbB, hB)) break;
    }
    // the last two chunks' sums
    for (int c = G - 2; c < G; ++c)
        if (ok && c >= 0) ok = mbar_wait_bounded(su32(&bar[c & 1]), (unsigned)(c >> 1) & 1u, timeout_ns);
    ok = __syncthreads_and(ok);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok) {
        for (int c = G - 2; c < G; ++c)
            if (c >= 0) drain_block(taddr, warp, c & 3, y);
        // warps 4-7 hand their low-half sums to warps 0-3 (same tile rows)
        // through the weight buffers, idle now that every MMA has finished
        float *lo = reinterpret_cast<float *>(A0);
        if (warp >= 4) {
#pragma unroll
            for (int n = 0; n < kTcTok; ++n) lo[n * kTcRows + (tid - kTcRows)] = y[n];
        }
    }
    __syncthreads();
    if (!ok) {
        if (tid == 0) atomicOr(err, kStatusTimeout);
    } else if (warp < 4) {
        // warps 0-3: tile row tid; y[n] = token row n's sum over all chunks
        const float *lo = reinterpret_cast<const float *>(A0);
#pragma unroll
        for (int n = 0; n < kTcTok; ++n) y[n] += lo[n * kTcRows + tid];
        const int r = kTcRows * tile + tid;
#pragma unroll 1
        for (int n = 0; n < nr; ++n) {
            float yn = 0.f;
#pragma unroll
            for (int t = 0; t < kTcTok; ++t) yn = t == n ? y[t] : yn;
            const int m = (int)__fns(mask, 0, n + 1);
            if constexpr (SWIGLU) {
                // rows 2j (gate) and 2j + 1 (up) of unit j = r / 2
                const float other = __shfl_xor_sync(0xFFFFFFFFu, yn, 1);
                if ((tid & 1) == 0 && m < M)
                    out[((size_t)u * M + m) * (rows / 2) + (r >> 1)] = yn / (1.0f + expf(-yn)) * other;
            } else {
                if (m < M) out[((size_t)u * M + m) * rows + r] = yn;
            }
        }
        (void)lane;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
}

// Two product sets in one grid (a second set lets the shared expert, with
// its own weights and code width, run beside the routed experts instead of
// after them): blockIdx.y < nA are slots of set a, the rest of set b;
// blockIdx.x is the 128-row tile.
template <int BITS_A, int BITS_B, bool SWIGLU>
__global__ void __launch_bounds__(kTcThreads, 2)
grouped_tc_kernel(const TcSet a, const TcSet b, int nA, int M, long long timeout_ns, int *err)
{
    const int y = blockIdx.y;
    if (y < nA) grouped_tc_body<BITS_A, SWIGLU>(a, y, blockIdx.x, M, timeout_ns, err);
    else grouped_tc_body<BITS_B, SWIGLU>(b, y - nA, blockIdx.x, M, timeout_ns, err);
}

}  // namespace

int launch_grouped_tc2(bool swiglu, int bits_a, const TcSetHost &ha, int nA, int bits_b, const TcSetHost *hb, int nB,
                       int M, int *err, long long timeout_ns, cudaStream_t stream)
{
    auto to_set = [](const TcSetHost &h) {
        return TcSet{h.W, h.rows, h.K, h.row_bytes, h.in, h.in_u, h.experts, h.masks, h.U_dev, h.out};
    };
    const TcSet a = to_set(ha);
    const TcSet b = hb ? to_set(*hb) : a;
    if (!hb) nB = 0;
    int tiles = ha.rows / kTcRows;
    if (hb && hb->rows / kTcRows > tiles) tiles = hb->rows / kTcRows;
    const dim3 grid((unsigned)tiles, (unsigned)(nA + nB));
    if (!hb) bits_b = bits_a;
    cudaError_t e = cudaErrorInvalidValue;
    auto go = [&](auto kernel) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e == cudaSuccess) kernel<<<grid, kTcThreads, kTcSmem, stream>>>(a, b, nA, M, timeout_ns, err);
    };
    // (a, b) code widths: both the same, or a routed width with 8-bit shared weights
    const int code = bits_a * 10 + bits_b;
    if (swiglu) {
        switch (code) {
        case 44: go(grouped_tc_kernel<4, 4, true>); break;
        case 66: go(grouped_tc_kernel<6, 6, true>); break;
        case 88: go(grouped_tc_kernel<8, 8, true>); break;
        case 48: go(grouped_tc_kernel<4, 8, true>); break;
        case 68: go(grouped_tc_kernel<6, 8, true>); break;
        default: return MOE_ERR_UNSUPPORTED;
        }
    } else {
        switch (code) {
        case 44: go(grouped_tc_kernel<4, 4, false>); break;
        case 66: go(grouped_tc_kernel<6, 6, false>); break;
        case 88: go(grouped_tc_kernel<8, 8, false>); break;
        case 48: go(grouped_tc_kernel<4, 8, false>); break;
        case 68: go(grouped_tc_kernel<6, 8, false>); break;
        default: return MOE_ERR_UNSUPPORTED;
        }
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        note_cuda_error((int)e);
        return MOE_ERR_CUDA;
    }
    note_launch();
    return MOE_OK;
}

int launch_grouped_tc(int bits, bool swiglu, const uint8_t *W, int rows, int K, int row_bytes, const float *in, int in_u,
                      int M, const int32_t *experts, const uint32_t *masks, int U, const int *U_dev, float *out,
                      int *err, long long timeout_ns, cudaStream_t stream)
{
    const TcSetHost h{W, rows, K, row_bytes, in, in_u, experts, masks, U_dev, out};
    return launch_grouped_tc2(swiglu, bits, h, U, bits, nullptr, 0, M, err, timeout_ns, stream);
}

int launch_gate_up_tc(const moe_layer &L, const float *hn, int M, const int32_t *experts, const uint32_t *masks, int U,
                      float *act, int *err, long long timeout_ns, cudaStream_t stream)
{
    const Geo &g = L.geo;
    return launch_grouped_tc(g.rb, true, L.ptrs.gu, 2 * g.I, g.H, g.g_bytes, hn, 0, M, experts, masks, U, nullptr, act,
                             err, timeout_ns, stream);
}

int launch_down_tc(const moe_layer &L, const float *act, int M, const int32_t *experts, const uint32_t *masks, int U,
                   float *y, int *err, long long timeout_ns, cudaStream_t stream)
{
    const Geo &g = L.geo;
    return launch_grouped_tc(g.rb, false, L.ptrs.down, g.H, g.I, g.d_bytes, act, M, M, experts, masks, U, nullptr, y,
                             err, timeout_ns, stream);
}

}  // namespace moe
