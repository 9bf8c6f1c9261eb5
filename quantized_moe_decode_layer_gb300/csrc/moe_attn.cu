// Decode attention with grouped query heads, split over the key axis, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory), for
// the attention shape of the 35B-A3B model: 16 query heads sharing 2
// key/value heads (8 per group), head dimension 256, bf16 key/value cache
// (PureDrive-35B-A3B-MLX model card, "How it works": one attention kernel for
// the one-row decode and the multi-row verify that reads K/V once for all
// query heads of a group and all verify rows, split over the keys
// flash-decoding style, with split points and summation order that depend
// only on the row's position; "Beyond this checkpoint": 16 query heads,
// 2 KV heads, head dim 256).
//
// What it computes: token row m (m < M) is at position pos0 + m and attends
// to keys 0 .. pos0 + m:
//     o[m][h] = sum_t softmax_t(q[m][h] . k[g][t] / 16) v[g][t],  g = h / 8.
//
// Split: the keys are cut into chunks of 512 positions (chunk j = keys
// 512 j .. 512 j + 511), the same for every row and every call; one CTA per
// (chunk, key/value head) computes, for every query column q = 8 m + head in
// group, the chunk's running maximum, the sum of exp(s - max) and the
// unnormalised sum of exp(s - max) v.  A second kernel merges a row's chunks
// in chunk order.  A row's result therefore depends only on its own position,
// query and the cache, never on M or on the other rows.
//
// Per CTA, over the chunk's tiles of 128 keys (warp-specialised):
//   - a TMA warp loads 16 KB boxes (128 rows x 64 bf16, 128-byte swizzle)
//     into a ring, one lane per box so that the boxes of a round go out
//     together: the tile's keys [128 keys x 256] in 4 boxes, then its values
//     from the transposed cache [256 d x 128 keys] in 4 boxes;
//   - an MMA warp issues S^T = K Q^T (M = 128 keys, N = the query columns,
//     K = 256 over d; Q in shared memory, written once) into one of two
//     tensor-memory score blocks, and O^T += V^T P^T (M = 128 values of d per
//     half, K = 128 keys) into the output block, with P in two bf16 halves
//     (p = hi + lo) stacked as the product's N columns (one instruction for
//     both: a tensor-core instruction of M = 128 costs about the same at any
//     N up to 256), so the weights keep ~16 significant bits;
//   - eight softmax warps read the score block (thread = key, every other
//     query column each, all columns' steps interleaved), mask keys past each row's position, take the
//     tile's column maxima (redux.sync on order-preserving keys) and the new
//     running maxima, write exp(s - max) as bf16 halves into shared memory
//     for the MMA and sum exactly those halves per column (all columns'
//     reductions interleaved, no branch between them); then they take the
//     previous tile's output block into fp32 registers (thread = one d of
//     one half), rescaled by exp(old max - new max) (online softmax).
//     (A tile of ones times the weights on the tensor core gave the column
//     sums too; it cost more in MMA instructions, the pipe that bounds a
//     tile, than the shuffles cost the softmax warps.)
// Every wait is bounded; one that runs out sets *err, the roles stop, the
// CTA waits (bounded) for its copies and MMAs and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <cstring>
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kAD = 256, kAHq = 16, kAHkv = 2, kAGrp = kAHq / kAHkv;
constexpr int kAKeys = 128;                 // keys per tile (MMA M of the score product)
constexpr int kATiles = 4;                  // tiles per chunk
constexpr int kAChunk = kAKeys * kATiles;   // keys per chunk: the split points are multiples of this
constexpr int kAMaxRows = 8;
constexpr int kAMaxPos = 1 << 19;           // cache positions at most (1024 chunks)
constexpr int kAMaxQ = kAGrp * kAMaxRows;   // query columns per key/value head
constexpr int kABox = 16384;                // one TMA box: 128 rows of 128 bytes
constexpr int kASoftWarps = 8;
constexpr int kASoftThreads = kASoftWarps * 32;
constexpr int kAThreads = kASoftThreads + 64;   // + TMA warp + MMA warp
// Tensor-memory columns: two score blocks of nq columns, then the output
// block (two halves of d, 2 nq columns each: the query columns of the high,
// then of the low weight halves). Up to 32 query columns this packs into 256
// columns, so that two CTAs fit on one SM; above, blocks sit at multiples of
// 64 and 128 in all 512.
__host__ __device__ constexpr bool tmem_compact(int nq) { return nq <= 32; }
__host__ __device__ constexpr uint32_t tmem_cols(int nq) { return tmem_compact(nq) ? 256u : 512u; }
__host__ __device__ constexpr uint32_t s_col(int nq, int b)
{
    return tmem_compact(nq) ? (uint32_t)(nq * b) : 64u * (uint32_t)b;
}
__host__ __device__ constexpr uint32_t o_col(int nq, int half)
{
    return tmem_compact(nq) ? (uint32_t)(2 * nq + 2 * nq * half) : 128u + 128u * (uint32_t)half;
}

struct AttnParams {
    CUtensorMap tk;   // keys: dims {256, n_valid, 2}, box {64, 128, 1}
    CUtensorMap tv;   // values, transposed: dims {n_valid, 256, 2}, box {64, 128, 1}
    const uint16_t *q;    // [M][16][256]
    float *part_o;        // [chunk][2][64][256]
    float *part_ml;       // [chunk][2][64][2]: running maximum, sum
    unsigned *seg_cnt;    // [M * 16] combine segments done (cleared by chunk CTA (0, 0))
    int M, pos0, n_valid, nq, nsub;
    long long timeout_ns;
    int *err;
};

// Shared-memory layout (offsets from a 1024-byte aligned base).
struct ALayout {
    int ring, q, p, red, bars, total;
};
__host__ __device__ inline ALayout attn_layout(int nq, int nsub)
{
    ALayout L;
    L.ring = 0;
    L.q = nsub * kABox;                       // Q: nq rows x 256, no swizzle, 4096 B per 8 rows
    L.p = L.q + nq * kAD * 2;                 // P: [2 buffers][hi, lo] nq rows x 128 keys
    L.red = L.p + 4 * nq * kAKeys * 2;        // reductions and running state
    L.bars = L.red + 4 * kAMaxQ * 4 * 2 + 4 * kAMaxQ * 4;
    L.total = L.bars + (2 * nsub + 11) * 8 + 16;
    return L;
}

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long gtime()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void bar_init(uint32_t b, unsigned n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t b)
{
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(b) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t b, unsigned bytes)
{
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(b), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool bar_test(uint32_t b, unsigned parity)
{
    uint32_t done;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(done)
                 : "r"(b), "r"(parity)
                 : "memory");
    return done != 0;
}

// Bounded wait on an mbarrier phase; gives up when the CTA's abort flag is
// set, or sets it (and the error word) when the time runs out.
__device__ __forceinline__ bool bar_wait(uint32_t b, unsigned parity, volatile int *abort, const AttnParams &p)
{
    if (bar_test(b, parity)) return true;
    const unsigned long long t0 = gtime();
#pragma unroll 1
    for (;;) {
        if (bar_test(b, parity)) return true;
        if (*abort) return false;
        if ((long long)(gtime() - t0) > p.timeout_ns) {
            *abort = 1;
            atomicOr(p.err, 1);
            return false;
        }
    }
}

// Named barrier of the softmax warps with an AND over their flags.
__device__ __forceinline__ bool soft_sync_and(bool ok)
{
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.and.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
                 : "=r"(r)
                 : "r"((uint32_t)ok), "r"(kASoftThreads)
                 : "memory");
    return r != 0;
}
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kASoftThreads) : "memory"); }

// Matrix descriptors (tcgen05 shared-memory descriptor, version 1).
// 128-byte swizzled K-major box (rows of 64 bf16, 8-row groups 1024 B apart):
// the K step of 16 elements advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
// No-swizzle K-major: 8 x 16-byte core matrices, 128 B apart along K, `sbo`
// bytes apart between 8-row groups.
__device__ __forceinline__ uint64_t desc_plain(uint32_t addr, uint32_t sbo)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = nq.
__device__ __forceinline__ uint32_t idesc_bf16(int nq)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nq >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t a, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(a)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// Order-preserving map of a float to an unsigned key and back.
__device__ __forceinline__ uint32_t fkey(float v)
{
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unkey(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k); }

// Element (r, k) of a no-swizzle K-major tile with 8-row groups `sbo` apart.
__device__ __forceinline__ uint32_t plain_off(int r, int k, uint32_t sbo)
{
    return (uint32_t)(r >> 3) * sbo + (uint32_t)(k >> 3) * 128u + (uint32_t)(r & 7) * 16u + (uint32_t)(k & 7) * 2u;
}

// Box j of a chunk of nt tiles, in ring order: tile 0's keys (4 boxes of
// 64 d), then for each tile t the keys of tile t + 1 (if any) and the
// values of tile t (4 boxes: half of d, then key half).
__device__ __forceinline__ void box_of(int j, int nt, bool &is_v, int &t, int &part)
{
    if (j < 4) { is_v = false; t = 0; part = j; return; }
    j -= 4;
    t = j >> 3;
    const int w = j & 7;
    if (t + 1 < nt && w < 4) { is_v = false; part = w; t = t + 1; }
    else { is_v = true; part = t + 1 < nt ? w - 4 : w; }
}

// MINB = 2: two CTAs per SM (at most 32 query columns, a shallower ring,
// registers capped at 96), for grids of more chunks than SMs.
template <int NQ, int MINB>
__global__ void __launch_bounds__(kAThreads, MINB) attn_chunk_kernel(const __grid_constant__ AttnParams p)
{
    constexpr int NC = NQ / 2;   // query columns of a softmax thread: q = 2 i + ch
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nsub = p.nsub, M = p.M, nreal = kAGrp * p.M;
    const ALayout L = attn_layout(NQ, nsub);
    const int chunk = blockIdx.x, g = blockIdx.y;
    const int k0 = chunk * kAChunk;
    const int nkeys = min(kAChunk, p.n_valid - k0);
    const int nt = (nkeys + kAKeys - 1) / kAKeys, nbox = 8 * nt;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the combine's segment counters of this call start at zero (the
    // combine kernel runs after this one on the stream)
    if (chunk == 0 && g == 0 && tid < M * kAHq) p.seg_cnt[tid] = 0u;

    uint8_t *ring = sm + L.ring, *qs = sm + L.q, *ps = sm + L.p;
    uint32_t *red_max = reinterpret_cast<uint32_t *>(sm + L.red);        // [4][64]
    float *red_sum = reinterpret_cast<float *>(red_max + 4 * kAMaxQ);    // [4][64]
    float *m_run = red_sum + 4 * kAMaxQ, *l_run = m_run + kAMaxQ;        // [64] each
    float *alpha = l_run + kAMaxQ;                                       // [2][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
    uint64_t *full = bars, *empty = bars + nsub;
    uint64_t *s_full = bars + 2 * nsub, *s_free = s_full + 2, *p_full = s_free + 2, *o_full = p_full + 2,
             *o_free = o_full + 1, *mma_done = o_free + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * nsub + 11);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    if (tid == 0) {
        for (int s = 0; s < nsub; ++s) {
            bar_init(su32(&full[s]), 1);
            bar_init(su32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(su32(&s_full[b]), 1);
            bar_init(su32(&s_free[b]), kASoftWarps);
            bar_init(su32(&p_full[b]), 1);
        }
        bar_init(su32(o_full), 1);
        bar_init(su32(o_free), kASoftWarps);
        bar_init(su32(mma_done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(tmem_cols(NQ))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Q of this key/value head as the score product's B operand: row
    // q = 8 m + head in group, zero past the last row
    for (int i = tid; i < NQ * (kAD / 8); i += kAThreads) {
        const int qr = i / (kAD / 8), dc = i % (kAD / 8);
        const int m = qr / kAGrp, hh = qr % kAGrp;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (m < M) v = __ldg(reinterpret_cast<const uint4 *>(p.q + ((size_t)m * kAHq + g * kAGrp + hh) * kAD) + dc);
        *reinterpret_cast<uint4 *>(qs + plain_off(qr, 8 * dc, 4096u)) = v;
    }
    for (int i = tid; i < kAMaxQ; i += kAThreads) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *tmem_slot;

    if (warp == kASoftWarps) {
        // ---------------------------------------------------------- TMA warp
        // batches of nsub boxes, one per lane: each lane waits for its own
        // slot to be released and issues, so the boxes go out together
        bool go = true;
#pragma unroll 1
        for (int base = 0; base < nbox && go; base += nsub) {
            const int j = base + lane;
            bool pending = lane < nsub && j < nbox;
            if (pending && base > 0 && !bar_wait(su32(&empty[lane]), (unsigned)((base / nsub) - 1) & 1u, abort_flag, p))
                pending = false;
            if (pending) {
                bool is_v;
                int t, part;
                box_of(j, nt, is_v, t, part);
                const uint32_t dst = su32(ring + (size_t)lane * kABox), fb = su32(&full[lane]);
                bar_expect(fb, kABox);
                const int kb = k0 + kAKeys * t;
                if (!is_v) tma_load3(dst, &p.tk, 64 * part, kb, g, fb);
                else tma_load3(dst, &p.tv, kb + 64 * (part & 1), 128 * (part >> 1), g, fb);
            }
            go = !__any_sync(0xFFFFFFFFu, *abort_flag != 0);
        }
        // every box issued must have landed before the CTA can exit: box j
        // of the last round of slot s
        const int rounds = (nbox + nsub - 1) / nsub;
        if (lane < nsub) {
            int last = -1;
            for (int r = rounds - 1; r >= 0 && last < 0; --r)
                if (r * nsub + lane < nbox) last = r;
            if (last >= 0) {
                const unsigned long long t0 = gtime();
                while (!bar_test(su32(&full[lane]), (unsigned)last & 1u) && (long long)(gtime() - t0) <= p.timeout_ns) {}
            }
        }
    } else if (warp == kASoftWarps + 1) {
        // ---------------------------------------------------------- MMA warp
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(NQ), id_o = idesc_bf16(2 * NQ);
            int slot = 0;
            unsigned ph = 0;
            bool go = true;
            auto take = [&]() -> bool {
                if (!go || !bar_wait(su32(&full[slot]), ph, abort_flag, p)) return go = false;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                return true;
            };
            auto release = [&]() {
                umma_commit(su32(&empty[slot]));
                if (++slot == nsub) { slot = 0; ph ^= 1u; }
            };
            auto scores = [&](int t) {
                const int b = t & 1;
                if (t >= 2 && !bar_wait(su32(&s_free[b]), (unsigned)((t - 2) >> 1) & 1u, abort_flag, p)) go = false;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                for (int part = 0; part < 4 && go; ++part) {
                    if (!take()) break;
                    const uint32_t a0 = su32(ring + (size_t)slot * kABox);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma(taddr + s_col(NQ, b), desc_sw128(a0 + 32u * k), desc_plain(su32(qs) + 256u * (4 * part + k), 4096u),
                             id_s, (part | k) != 0 ? 1u : 0u);
                    release();
                }
                if (go) umma_commit(su32(&s_full[b]));
            };
            // O^T += V^T [P_hi; P_lo]^T: the two halves of the weights are the
            // columns 0 .. NQ - 1 and NQ .. 2 NQ - 1 of one product
            auto values = [&](int t) {
                const int b = t & 1;
                if (!bar_wait(su32(&p_full[b]), (unsigned)(t >> 1) & 1u, abort_flag, p)) go = false;
                if (go && t >= 1 && !bar_wait(su32(o_free), (unsigned)(t - 1) & 1u, abort_flag, p)) go = false;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t pb = su32(ps) + (uint32_t)b * (uint32_t)(2 * NQ * kAKeys * 2);
                for (int part = 0; part < 4 && go; ++part) {
                    if (!take()) break;
                    const int half = part >> 1, kh = part & 1;
                    const uint32_t a0 = su32(ring + (size_t)slot * kABox);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t bd = desc_plain(pb + 256u * (4 * kh + k), 2048u);
                        umma(taddr + o_col(NQ, half), desc_sw128(a0 + 32u * k), bd, id_o, (kh | k) != 0 ? 1u : 0u);
                    }
                    release();
                }
                if (go) umma_commit(su32(o_full));
            };
            scores(0);
            for (int t = 0; t < nt && go; ++t) {
                if (t + 1 < nt) scores(t + 1);
                if (go) values(t);
            }
            // every MMA issued has finished before the tensor memory is freed
            umma_commit(su32(mma_done));
            const unsigned long long t0 = gtime();
            while (!bar_test(su32(mma_done), 0u) && (long long)(gtime() - t0) <= p.timeout_ns) {}
        }
    } else {
        // ------------------------------------------------------ softmax warps
        // thread = key 32 qt + lane of a tile (columns q = 2 i + ch), and, for
        // the output, d = 128 ch + 32 qt + lane
        const int qt = warp & 3, ch = warp >> 2;
        const int key_local = 32 * qt + lane;
        const int dl = 128 * ch + 32 * qt + lane;
        float oacc[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) oacc[i] = 0.f;
        bool ok = true;
        auto drain = [&](int t) {
            ok = __all_sync(0xFFFFFFFFu, bar_wait(su32(o_full), (unsigned)t & 1u, abort_flag, p));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!ok) return;
            const uint32_t base = taddr + ((uint32_t)(32 * qt) << 16) + o_col(NQ, ch);
            const float *al = alpha + (t & 1) * kAMaxQ;
            // columns q (high halves) and NQ + q (low halves), 8 at a time
#pragma unroll
            for (int c8 = 0; c8 < NQ / 8; ++c8) {
                float hi[8], lo[8];
                tmem_ld8(base + 8u * c8, hi);
                tmem_ld8(base + (uint32_t)NQ + 8u * c8, lo);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) oacc[8 * c8 + i] = fmaf(oacc[8 * c8 + i], al[8 * c8 + i], hi[i] + lo[i]);
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) bar_arrive(su32(o_free));
        };
#pragma unroll 1
        for (int t = 0; t < nt; ++t) {
            const int b = t & 1;
            const int key = k0 + kAKeys * t + key_local;
            ok = __all_sync(0xFFFFFFFFu, bar_wait(su32(&s_full[b]), (unsigned)(t >> 1) & 1u, abort_flag, p));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            float sv[NC];
            if (ok) {
                const uint32_t base = taddr + ((uint32_t)(32 * qt) << 16) + s_col(NQ, b);
                // 16 columns at a time, keeping every other one (q = 2 i + ch)
#pragma unroll
                for (int c16 = 0; c16 < NQ / 16; ++c16) {
                    float w0[8], w1[8];
                    tmem_ld8(base + 16u * c16, w0);
                    tmem_ld8(base + 16u * c16 + 8u, w1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        sv[8 * c16 + i] = w0[2 * i + ch];
                        sv[8 * c16 + 4 + i] = w1[2 * i + ch];
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) bar_arrive(su32(&s_free[b]));
            }
            if (!soft_sync_and(ok)) { ok = false; break; }
            // scale and mask (key valid for row m when key <= pos0 + m), then
            // the tile's column maxima over the warp's keys
            uint32_t mk[NC];
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int q = 2 * i + ch, m = q >> 3;
                const bool valid = q < nreal && key <= p.pos0 + m && key < p.n_valid;
                sv[i] = valid ? sv[i] * 0.0625f : -INFINITY;
                mk[i] = fkey(sv[i]);
            }
            // (every column, padding included: branches around the
            // reductions would keep them from overlapping)
#pragma unroll
            for (int i = 0; i < NC; ++i) mk[i] = __reduce_max_sync(0xFFFFFFFFu, mk[i]);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < NC; ++i) red_max[qt * kAMaxQ + 2 * i + ch] = mk[i];
            }
            soft_sync();
            // new running maxima, then exp(s - max) as bf16 halves into P
            // (rows q and NQ + q of the value product's B operand, key along
            // K) and the column sums of what the MMA sees
            float mnew[NC];
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int q = 2 * i + ch;
                const uint32_t a = max(red_max[q], red_max[kAMaxQ + q]);
                const uint32_t c = max(red_max[2 * kAMaxQ + q], red_max[3 * kAMaxQ + q]);
                mnew[i] = fmaxf(m_run[q], unkey(max(a, c)));
            }
            uint8_t *pbuf = ps + (size_t)b * (size_t)(2 * NQ * kAKeys * 2);
#pragma unroll
            for (int i = 0; i < NC; ++i) {
                const int q = 2 * i + ch;
                const float e = sv[i] == -INFINITY ? 0.f : expf(sv[i] - mnew[i]);
                const __nv_bfloat16 h = __float2bfloat16_rn(e);
                const __nv_bfloat16 lo = __float2bfloat16_rn(e - __bfloat162float(h));
                *reinterpret_cast<__nv_bfloat16 *>(pbuf + plain_off(q, key_local, 2048u)) = h;
                *reinterpret_cast<__nv_bfloat16 *>(pbuf + plain_off(NQ + q, key_local, 2048u)) = lo;
                sv[i] = __bfloat162float(h) + __bfloat162float(lo);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                for (int i = 0; i < NC; ++i) sv[i] += __shfl_xor_sync(0xFFFFFFFFu, sv[i], o);
            if (lane == 0) {
#pragma unroll
                for (int i = 0; i < NC; ++i) red_sum[qt * kAMaxQ + 2 * i + ch] = sv[i];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            soft_sync();
            if (tid == 0) bar_arrive(su32(&p_full[b]));
            if (tid < NQ) {
                const int q = tid;
                const uint32_t a = max(red_max[q], red_max[kAMaxQ + q]);
                const uint32_t c = max(red_max[2 * kAMaxQ + q], red_max[3 * kAMaxQ + q]);
                const float mold = m_run[q], mn = fmaxf(mold, unkey(max(a, c)));
                const float al = mn == -INFINITY ? 1.f : expf(mold - mn);
                const float lt = ((red_sum[q] + red_sum[kAMaxQ + q]) + red_sum[2 * kAMaxQ + q]) + red_sum[3 * kAMaxQ + q];
                l_run[q] = fmaf(l_run[q], al, lt);
                m_run[q] = mn;
                alpha[b * kAMaxQ + q] = al;
            }
            if (t >= 1) {
                drain(t - 1);
                if (!soft_sync_and(ok)) { ok = false; break; }
            }
        }
        if (ok && nt >= 1) {
            soft_sync();   // the last tile's alpha is written
            drain(nt - 1);
        }
        ok = soft_sync_and(ok);
        if (ok) {
            const size_t cg = (size_t)chunk * kAHkv + g;
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                if (q < nreal) p.part_o[(cg * kAMaxQ + q) * kAD + dl] = oacc[q];
            if (tid < nreal) {
                p.part_ml[(cg * kAMaxQ + tid) * 2] = m_run[tid];
                p.part_ml[(cg * kAMaxQ + tid) * 2 + 1] = l_run[tid];
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(tmem_cols(NQ)) : "memory");
}

// Merge of a row's chunks, in chunk order: o = sum_j e^(m_j - M) O_j /
// sum_j e^(m_j - M) l_j with M the largest chunk maximum.  One CTA per
// (row, query head), thread = d.  The chunk maxima and weights go through
// shared memory (all threads load them together), then each thread's loads
// of its d from every chunk are independent and overlap.
constexpr int kACombineChunks = kAMaxPos / kAChunk;
constexpr int kASeg = 16;                               // chunks per combine segment

// The chunks of row m, head h merged: every chunk's output rescaled by
// exp(its running maximum - the maximum over all chunks) and summed, and
// divided by the sum of its rescaled sums.  One CTA per (row, head, segment
// of kASeg chunks): each sums its segment in chunk order (thread = d); the
// last CTA of a (row, head) to finish (a counter, after a memory fence)
// adds the segments' sums in segment order.  The order depends only on the
// row's position, so a row's result does not depend on M.
__global__ void __launch_bounds__(kAD) attn_combine_kernel(const float *part_o, const float *part_ml, int pos0,
                                                           float *o, float *seg_o, float *seg_l, unsigned *seg_cnt,
                                                           int smax)
{
    __shared__ float wsh[kASeg];
    __shared__ float red[kAD / 32];
    __shared__ int last;
    const int mh = blockIdx.x, seg = blockIdx.y;
    const int m = mh / kAHq, h = mh % kAHq, g = h / kAGrp, q = kAGrp * m + h % kAGrp;
    const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
    const int J = (pos0 + m + 1 + kAChunk - 1) / kAChunk;   // <= kACombineChunks (host check)
    const int S = (J + kASeg - 1) / kASeg;
    if (seg >= S) return;
    auto ml = [&](int j) { return part_ml + (((size_t)j * kAHkv + g) * kAMaxQ + q) * 2; };
    float mx = -INFINITY;
    for (int j = d; j < J; j += kAD) mx = fmaxf(mx, __ldg(ml(j)));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kAD / 32; ++w) mx = fmaxf(mx, red[w]);
    const int j0 = seg * kASeg, nj = min(kASeg, J - j0);
    if (d < nj) wsh[d] = expf(__ldg(ml(j0 + d)) - mx);
    __syncthreads();
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int jj = 0; jj < kASeg; ++jj)
        if (jj < nj) {
            const size_t c = ((size_t)(j0 + jj) * kAHkv + g) * kAMaxQ + q;
            const float w = wsh[jj];
            lsum = fmaf(__ldg(part_ml + 2 * c + 1), w, lsum);
            acc = fmaf(__ldg(part_o + c * kAD + d), w, acc);
        }
    float *out = o + ((size_t)m * kAHq + h) * kAD + d;
    if (S == 1) {
        *out = acc / lsum;
        return;
    }
    seg_o[((size_t)mh * smax + seg) * kAD + d] = acc;
    if (d == 0) seg_l[(size_t)mh * smax + seg] = lsum;
    __threadfence();
    __syncthreads();
    if (d == 0) last = atomicAdd(seg_cnt + mh, 1u) == (unsigned)(S - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();
    float a = 0.f, l = 0.f;
#pragma unroll 4
    for (int s2 = 0; s2 < S; ++s2) {
        a += __ldcg(seg_o + ((size_t)mh * smax + s2) * kAD + d);
        l += __ldcg(seg_l + (size_t)mh * smax + s2);
    }
    *out = a / l;
}

// New rows' keys and values into the cache: row m at position pos0 + m;
// values go to the transposed cache.  One CTA per (row, key/value head).
__global__ void __launch_bounds__(kAD) attn_append_kernel(const uint16_t *kn, const uint16_t *vn, int pos0,
                                                          uint16_t *kc, uint16_t *vtc, int T_cap)
{
    const int m = blockIdx.x / kAHkv, g = blockIdx.x % kAHkv, d = threadIdx.x, t = pos0 + m;
    kc[((size_t)g * T_cap + t) * kAD + d] = kn[((size_t)m * kAHkv + g) * kAD + d];
    vtc[((size_t)g * kAD + d) * T_cap + t] = vn[((size_t)m * kAHkv + g) * kAD + d];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

int attn_max_positions() { return kAMaxPos; }

// Workspace: per-chunk maxima and sums [chunk][2][64][2], per-chunk outputs
// [chunk][2][64][256], the combine's segment sums [8 * 16][seg] and segment
// outputs [8 * 16][seg][256], and its counters [8 * 16] (fp32 / u32, each
// region 256-byte aligned).
struct AWs {
    size_t ml, po, sl, so, cnt, total;
    int smax;
};
AWs attn_ws_layout(int T_cap)
{
    AWs w;
    const size_t nchunks = (size_t)(T_cap + kAChunk - 1) / kAChunk;
    w.smax = (int)((nchunks + kASeg - 1) / kASeg);
    const size_t mh = (size_t)kAMaxRows * kAHq;
    w.ml = 0;
    w.po = align_up(nchunks * kAHkv * kAMaxQ * 2 * sizeof(float), 256);
    w.sl = align_up(w.po + nchunks * kAHkv * kAMaxQ * kAD * sizeof(float), 256);
    w.so = align_up(w.sl + mh * w.smax * sizeof(float), 256);
    w.cnt = align_up(w.so + mh * w.smax * kAD * sizeof(float), 256);
    w.total = align_up(w.cnt + mh * sizeof(unsigned), 256);
    return w;
}

size_t attn_workspace_bytes(int T_cap) { return attn_ws_layout(T_cap).total; }

int launch_attn(const uint16_t *q, const uint16_t *k, const uint16_t *vt, int T_cap, int pos0, int M, float *o,
                void *ws, int *err, long long timeout_ns, cudaStream_t stream)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return MOE_ERR_UNSUPPORTED;
    const int n_valid = pos0 + M, nchunks = (n_valid + kAChunk - 1) / kAChunk;
    AttnParams P;
    memset(&P, 0, sizeof P);
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kAD, (cuuint64_t)n_valid, (cuuint64_t)kAHkv};
        const cuuint64_t strides[2] = {(cuuint64_t)kAD * 2, (cuuint64_t)T_cap * kAD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kAKeys, 1}, es[3] = {1, 1, 1};
        if (enc(&P.tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(k), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_INVALID_ARG;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)n_valid, (cuuint64_t)kAD, (cuuint64_t)kAHkv};
        const cuuint64_t strides[2] = {(cuuint64_t)T_cap * 2, (cuuint64_t)kAD * T_cap * 2};
        const cuuint32_t box[3] = {64, 128, 1}, es[3] = {1, 1, 1};
        if (enc(&P.tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(vt), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return MOE_ERR_INVALID_ARG;
    }
    const size_t nchunks_cap = (size_t)(T_cap + kAChunk - 1) / kAChunk;
    P.q = q;
    const AWs aw = attn_ws_layout(T_cap);
    P.seg_cnt = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(ws) + aw.cnt);
    P.part_ml = static_cast<float *>(ws);
    P.part_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) +
                                         align_up(nchunks_cap * kAHkv * kAMaxQ * 2 * sizeof(float), 256));
    P.M = M;
    P.pos0 = pos0;
    P.n_valid = n_valid;
    P.nq = 16 * ((kAGrp * M + 15) / 16);
    P.timeout_ns = timeout_ns;
    P.err = err;
    static std::once_flag attr_once[64];
    static int sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    std::call_once(attr_once[dev], [&] {
        const void *fns[6] = {(const void *)attn_chunk_kernel<16, 1>, (const void *)attn_chunk_kernel<32, 1>,
                              (const void *)attn_chunk_kernel<48, 1>, (const void *)attn_chunk_kernel<64, 1>,
                              (const void *)attn_chunk_kernel<16, 2>, (const void *)attn_chunk_kernel<32, 2>};
        for (int i = 0; i < 6 && e == cudaSuccess; ++i) {
            e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(fns[i], cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
        }
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    });
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    // More chunk CTAs than SMs: two per SM when the tensor memory and a
    // shallower ring allow it (16 query columns: 5 boxes, 32: 3, within
    // half of the SM's shared memory); otherwise one per SM with 8 boxes.
    const bool two_per_sm = tmem_compact(P.nq) && (long long)nchunks * kAHkv > sm_count[dev];
    if (two_per_sm)
        P.nsub = P.nq <= 16 ? 5 : 3;
    else
        P.nsub = attn_layout(P.nq, 8).total + 1024 <= kSmemMax ? 8 : 6;
    const int smem = attn_layout(P.nq, P.nsub).total + 1024;
    if (smem > kSmemMax) return MOE_ERR_UNSUPPORTED;
    const dim3 grid(nchunks, kAHkv);
    if (two_per_sm) {
        if (P.nq == 16) attn_chunk_kernel<16, 2><<<grid, kAThreads, smem, stream>>>(P);
        else attn_chunk_kernel<32, 2><<<grid, kAThreads, smem, stream>>>(P);
    } else {
        switch (P.nq) {
        case 16: attn_chunk_kernel<16, 1><<<grid, kAThreads, smem, stream>>>(P); break;
        case 32: attn_chunk_kernel<32, 1><<<grid, kAThreads, smem, stream>>>(P); break;
        case 48: attn_chunk_kernel<48, 1><<<grid, kAThreads, smem, stream>>>(P); break;
        default: attn_chunk_kernel<64, 1><<<grid, kAThreads, smem, stream>>>(P); break;
        }
    }
    note_launch();
    {
        // segments of the last row (the most chunks); other rows' CTAs past
        // their own segments return at once
        const int Jmax = (pos0 + M + kAChunk - 1) / kAChunk;
        const dim3 cgrid(M * kAHq, (Jmax + kASeg - 1) / kASeg);
        attn_combine_kernel<<<cgrid, kAD, 0, stream>>>(
            P.part_o, P.part_ml, pos0, o, reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + aw.so),
            reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + aw.sl), P.seg_cnt, aw.smax);
    }
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

int launch_attn_append(const uint16_t *kn, const uint16_t *vn, int M, int pos0, uint16_t *kc, uint16_t *vtc, int T_cap,
                       cudaStream_t stream)
{
    attn_append_kernel<<<M * kAHkv, kAD, 0, stream>>>(kn, vn, pos0, kc, vtc, T_cap);
    note_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

}  // namespace moe
