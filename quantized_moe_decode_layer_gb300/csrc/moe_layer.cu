// Persistent decode kernel of the quantized MoE FFN layer (and of a stack of
// such layers) for sm_103a.
//
// One CTA per SM; 8 compute warps and 1 producer warp per CTA.  The producer
// streams every weight byte the CTA needs through a ring of shared-memory
// stages with 1-D bulk copies (cp.async.bulk + mbarrier transaction counts);
// the compute warps dequantise in registers and accumulate in fp32.  Per layer:
//
//   P0  every CTA: RMSNorm of the M input rows into shared memory
//       (flash-moe, "Metal Compute Shaders": RMS normalisation)
//   P1  router rows (and the shared-expert gate row) and the shared expert's
//       gate/up units, split evenly over the CTAs            -> grid barrier
//   R   every CTA: softmax + top-k + renormalisation per row, then the list
//       of distinct selected experts with the rows that chose each
//       (PureDrive model card, "Summary": full top-8 of 256)
//   P2  gate/up units of the selected experts, each expert streamed once for
//       all the rows that chose it (model card, "How it works": the verify
//       pass reads its weights once), SwiGLU                 -> grid barrier
//   P3  each CTA owns a slice of the H outputs: down rows of every selected
//       expert and of the shared expert, weighted combine, sigmoid-gated
//       shared expert and residual (flash-moe: "MoE combine + residual +
//       gate"); rows of the next layer's weights keep streaming meanwhile
//                                                             -> grid barrier
//   N   the fused next RMSNorm of the bf16 output (model card: fused
//       add+RMSNorm), or the next layer's P0.
//
// Determinism: no float atomics; every sum has a fixed order that depends
// only on the row itself, so row m of an M-row call equals a 1-row call.
#include <cuda_bf16.h>

#include <cfloat>
#include <cstdio>

#include "moe_internal.h"
#include "moe_unpack.cuh"

namespace moe {
namespace {

constexpr int NCW = kConsumerWarps;
constexpr int NCT = NCW * 32;
constexpr int kCandCap = 64;
constexpr unsigned FULLMASK = 0xffffffffu;

// ------------------------------------------------------------ shared layout

struct SmemLayout {
    int bar, flags, slot_e, slot_mask, slot_rowbase, slot_w, sigma, eslot, emask, topv, tope, topw;
    int cand_v, cand_e, pair_slot, pair_m, red, xs, xsum, acc, ring, total;
};

__host__ __device__ inline int take(int &o, int bytes, int align)
{
    o = (int)align_up((size_t)o, (size_t)align);
    const int r = o;
    o += bytes;
    return r;
}

__host__ __device__ inline SmemLayout carve(const Geo &g, const Plan &p)
{
    SmemLayout L;
    int o = 0;
    const int ms = p.max_slots;
    L.bar = take(o, (2 * p.NS + 1) * 8, 8);
    L.flags = take(o, 16 * 4, 16);
    L.slot_e = take(o, ms * 4, 4);
    L.slot_mask = take(o, ms * 4, 4);
    L.slot_rowbase = take(o, (ms + 1) * 4, 4);
    L.slot_w = take(o, ms * kMaxRows * 4, 4);
    L.sigma = take(o, kMaxRows * 4, 4);
    L.eslot = take(o, g.E * 4, 4);
    L.emask = take(o, g.E * 4, 4);
    L.topv = take(o, kMaxRows * kMaxK * 4, 4);
    L.tope = take(o, kMaxRows * kMaxK * 4, 4);
    L.topw = take(o, kMaxRows * kMaxK * 4, 4);
    L.cand_v = take(o, NCW * kCandCap * 4, 4);
    L.cand_e = take(o, NCW * kCandCap * 4, 4);
    L.pair_slot = take(o, ms * kMaxRows * 4, 4);
    L.pair_m = take(o, ms * kMaxRows * 4, 4);
    L.red = take(o, (NCW + 2) * kMaxRows * 4, 4);
    L.xs = take(o, p.maxr * g.H * 4, 16);
    L.xsum = take(o, p.maxr * (g.H / kSub) * 4, 16);
    L.acc = take(o, p.hrows * kMaxRows * 4, 16);
    L.ring = take(o, p.NS * p.S, 128);
    L.total = o;
    return L;
}

__host__ __device__ inline int lanes_per_row(int K) { return K / kSub < 32 ? K / kSub : 32; }

// ------------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned tx)
{
    [[maybe_unused]] uint64_t st;
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(st) : "r"(smem_u32(bar)), "r"(tx) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar, unsigned count)
{
    [[maybe_unused]] uint64_t st;
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(st) : "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ unsigned long long now_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Named barrier over the compute warps only, with an OR-reduction.
__device__ __forceinline__ bool cbar_or(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred pi, po;\n\t"
                 "setp.ne.u32 pi, %1, 0;\n\t"
                 "bar.red.or.pred po, 1, %2, pi;\n\t"
                 "selp.u32 %0, 1, 0, po;\n\t}"
                 : "=r"(r) : "r"((uint32_t)v), "n"(NCT) : "memory");
    return r != 0;
}

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

__device__ __forceinline__ unsigned atom_add_acqrel(unsigned *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(unsigned *p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf(float v)
{
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(FULLMASK, v, o);
    return v;
}

// ----------------------------------------------------------- CTA state

struct Sh {
    uint64_t *full, *empty, *route;
    int *flags;          // [0] abort, [1] U
    int *slot_e;
    uint32_t *slot_mask;
    int *slot_rowbase;
    float *slot_w;       // [slot][kMaxRows]
    float *sigma;        // [kMaxRows]
    int *eslot;
    uint32_t *emask;
    float *topv;         // [kMaxRows][kMaxK]
    int *tope;
    float *topw;
    float *cand_v;       // [NCW][kCandCap]
    int *cand_e;
    int *pair_slot, *pair_m;
    float *red;          // [(NCW + 2) * kMaxRows]
    float *xs;           // arranged activations (hn in P0..P2, act chunks in P3)
    float *xsum;         // per-16 sums of xs
    float *acc;          // [hrows][kMaxRows] output accumulators
    uint8_t *ring;
    int NS, S;
    long long timeout_ns;
    Ctrl *ctrl;
};

__device__ __forceinline__ bool aborted(const Sh &sh) { return *(volatile int *)&sh.flags[0] != 0; }

__device__ void raise_abort(const Sh &sh, int where)
{
    *(volatile int *)&sh.flags[0] = 1;
    atomicOr(&sh.ctrl->status, kStatusTimeout);
    atomicExch(&sh.ctrl->where, where);
}

// Bounded wait on an mbarrier phase; false on timeout or abort.
__device__ bool wait_bar(const Sh &sh, uint64_t *bar, unsigned parity, int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (aborted(sh)) return false;
            if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) {
                raise_abort(sh, where);
                return false;
            }
        }
    }
}

// Grid-wide barrier over the compute warps of every CTA (bounded spin).
__device__ bool grid_sync(const KParams &kp, const Sh &sh, unsigned &gen, int &nsync)
{
    if (cbar_or(aborted(sh))) return false;
    if (threadIdx.x == 0) {
        Ctrl *ctrl = sh.ctrl;
        const bool skip = kp.skip_cta == (int)blockIdx.x && nsync == 0;
        bool released = false;
        if (!skip) {
            const unsigned old = atom_add_acqrel(&ctrl->count, 1u);
            if (old == gridDim.x - 1) {
                st_relaxed(&ctrl->count, 0u);
                st_release(&ctrl->gen, gen + 1);
                released = true;
            }
        }
        if (!released) {
            const unsigned long long t0 = now_ns();
            for (unsigned it = 0;; ++it) {
                if (ld_acquire(&ctrl->gen) != gen) break;
                if ((it & 63) == 63) {
                    if (*(volatile int *)&ctrl->status != 0) { *(volatile int *)&sh.flags[0] = 1; break; }
                    if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) { raise_abort(sh, 100 + nsync); break; }
                }
            }
        }
        gen += 1;
        nsync += 1;
    }
    return !cbar_or(aborted(sh));
}

__device__ __forceinline__ void split(int n, int P, int c, int &a, int &b)
{
    a = (int)((long long)n * c / P);
    b = (int)((long long)n * (c + 1) / P);
}

// ------------------------------------------------------ dot-product kernels

// Arranged float4 index of (sub-group sg, quarter t) for vectors of K inputs:
// lanes holding consecutive sub-groups read consecutive float4s.
__device__ __forceinline__ int arr_index(int sg, int t, int LPR)
{
    return (sg / LPR) * 4 * LPR + t * LPR + (sg % LPR);
}

template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t *row, int sg, uint32_t (&w)[4])
{
    if (BITS == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + sg * 8);
        w[0] = v.x; w[1] = v.y;
    } else if (BITS == 6) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(row + sg * 12);
        w[0] = p[0]; w[1] = p[1]; w[2] = p[2];
    } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + sg * 16);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
}

template <int BITS, int T>
__device__ __forceinline__ void get4(const uint32_t (&w)[4], float (&q)[4])
{
    Unpack<BITS>::template get4<T>(w, q);
}

// One quarter (4 codes) of a sub-group: S[n][r] += sum_i q[n][i] * x[r][i].
template <int BITS, int NR, int NW, int T>
__device__ __forceinline__ void quarter(const uint32_t (&w)[NW][4], const float4 *xs4, const int (&xoff)[NR],
                                        int ai, int LPR, float (&S0)[NW][NR], float (&S1)[NW][NR])
{
    float q[NW][4];
#pragma unroll
    for (int n = 0; n < NW; ++n) get4<BITS, T>(w[n], q[n]);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float4 x = xs4[xoff[r] + ai + T * LPR];
#pragma unroll
        for (int n = 0; n < NW; ++n) {
            S0[n][r] = fmaf(q[n][0], x.x, S0[n][r]);
            S1[n][r] = fmaf(q[n][1], x.y, S1[n][r]);
            S0[n][r] = fmaf(q[n][2], x.z, S0[n][r]);
            S1[n][r] = fmaf(q[n][3], x.w, S1[n][r]);
        }
    }
}

// Sub-group sg (16 inputs) of NW weight rows against NR activation vectors:
// acc[n][r] += s_g * sum(q x) + b_g * sum(x)  (per-group affine factoring of
// sum_j (q_j s + b) x_j).
template <int BITS, int NR, int NW>
__device__ __forceinline__ void qdot_sub(const uint8_t *const (&wr)[NW], int K, int sg, const float4 *xs4,
                                         const float *xsum, const int (&xoff)[NR], const int (&soff)[NR],
                                         int LPR, float (&acc)[NW][NR])
{
    const int ai = arr_index(sg, 0, LPR);
    if constexpr (BITS == 0) {
        // fp32 rows
#pragma unroll
        for (int n = 0; n < NW; ++n) {
            const float4 *wp = reinterpret_cast<const float4 *>(wr[n] + sg * 64);
            float S[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) S[r] = 0.f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 wv = wp[t];
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const float4 x = xs4[xoff[r] + ai + t * LPR];
                    S[r] = fmaf(wv.x, x.x, S[r]);
                    S[r] = fmaf(wv.y, x.y, S[r]);
                    S[r] = fmaf(wv.z, x.z, S[r]);
                    S[r] = fmaf(wv.w, x.w, S[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[n][r] += S[r];
        }
        return;
    } else {
        uint32_t w[NW][4];
        float s[NW], b[NW];
#pragma unroll
        for (int n = 0; n < NW; ++n) {
            load_codes<BITS>(wr[n], sg, w[n]);
            const uint32_t sbw = *reinterpret_cast<const uint32_t *>(wr[n] + K * BITS / 8 + (sg >> 2) * 4);
            s[n] = __uint_as_float(sbw << 16);
            b[n] = __uint_as_float(sbw & 0xFFFF0000u);
        }
        float S0[NW][NR], S1[NW][NR];
#pragma unroll
        for (int n = 0; n < NW; ++n)
#pragma unroll
            for (int r = 0; r < NR; ++r) S0[n][r] = S1[n][r] = 0.f;
        quarter<BITS, NR, NW, 0>(w, xs4, xoff, ai, LPR, S0, S1);
        quarter<BITS, NR, NW, 1>(w, xs4, xoff, ai, LPR, S0, S1);
        quarter<BITS, NR, NW, 2>(w, xs4, xoff, ai, LPR, S0, S1);
        quarter<BITS, NR, NW, 3>(w, xs4, xoff, ai, LPR, S0, S1);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float xsm = xsum[soff[r] + sg];
#pragma unroll
            for (int n = 0; n < NW; ++n) {
                acc[n][r] = fmaf(s[n], S0[n][r] + S1[n][r], acc[n][r]);
                acc[n][r] = fmaf(b[n], xsm, acc[n][r]);
            }
        }
    }
}

template <int NR>
__device__ __forceinline__ void rows_from_mask(uint32_t mask, int (&rows)[NR], int &nvalid)
{
    nvalid = 0;
    int last = 0;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        if (mask) {
            last = __ffs(mask) - 1;
            mask &= mask - 1;
            ++nvalid;
        }
        rows[r] = last;
    }
}

// Gate/up units (gate row, up row) of one stage -> act[m * mstride + j0 + u].
template <int BITS, int NR>
__device__ void gu_stage(const Sh &sh, const uint8_t *stage, int cnt, int rowb, int H, uint32_t mask,
                         float *act, int mstride, int j0)
{
    const int lane = threadIdx.x & 31;
    const int LPR = lanes_per_row(H), RPP = 32 / LPR, nsg = H / kSub;
    int rows[NR], nvalid;
    rows_from_mask<NR>(mask, rows, nvalid);
    int xoff[NR], soff[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) { xoff[r] = rows[r] * (H / 4); soff[r] = rows[r] * nsg; }
    const float4 *xs4 = reinterpret_cast<const float4 *>(sh.xs);
    for (int u0 = 0; u0 < cnt; u0 += RPP) {
        const int u = u0 + lane / LPR;
        const bool valid = u < cnt;
        float acc[2][NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[0][r] = acc[1][r] = 0.f;
        if (valid) {
            const uint8_t *const wr[2] = {stage + (size_t)u * 2 * rowb, stage + (size_t)u * 2 * rowb + rowb};
            for (int sg = lane % LPR; sg < nsg; sg += LPR)
                qdot_sub<BITS, NR, 2>(wr, H, sg, xs4, sh.xsum, xoff, soff, LPR, acc);
        }
        for (int o = LPR / 2; o >= 1; o >>= 1)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                acc[0][r] += __shfl_xor_sync(FULLMASK, acc[0][r], o);
                acc[1][r] += __shfl_xor_sync(FULLMASK, acc[1][r], o);
            }
        if (valid && lane % LPR == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
                if (r < nvalid) {
                    const float g = acc[0][r], up = acc[1][r];
                    act[(size_t)rows[r] * mstride + j0 + u] = g / (1.0f + expf(-g)) * up;
                }
        }
    }
}

// Router rows of one stage -> logits[m * Er + e0 + u].
template <int BITS, int NR>
__device__ void router_stage(const Sh &sh, const uint8_t *stage, int cnt, int rowb, int H, uint32_t mask,
                             float *logits, int Er, int e0)
{
    const int lane = threadIdx.x & 31;
    const int LPR = lanes_per_row(H), RPP = 32 / LPR, nsg = H / kSub;
    int rows[NR], nvalid;
    rows_from_mask<NR>(mask, rows, nvalid);
    int xoff[NR], soff[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) { xoff[r] = rows[r] * (H / 4); soff[r] = rows[r] * nsg; }
    const float4 *xs4 = reinterpret_cast<const float4 *>(sh.xs);
    for (int u0 = 0; u0 < cnt; u0 += RPP) {
        const int u = u0 + lane / LPR;
        const bool valid = u < cnt;
        float acc[1][NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[0][r] = 0.f;
        if (valid) {
            const uint8_t *const wr[1] = {stage + (size_t)u * rowb};
            for (int sg = lane % LPR; sg < nsg; sg += LPR)
                qdot_sub<BITS, NR, 1>(wr, H, sg, xs4, sh.xsum, xoff, soff, LPR, acc);
        }
        for (int o = LPR / 2; o >= 1; o >>= 1)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[0][r] += __shfl_xor_sync(FULLMASK, acc[0][r], o);
        if (valid && lane % LPR == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
                if (r < nvalid) logits[(size_t)rows[r] * Er + e0 + u] = acc[0][r];
        }
    }
}

// Down rows [rs, rs + cnt) (relative to the CTA's first output) of one
// expert; the warp handles the rows it owns (row % NCW == warp) and adds
// wgt[m] * y into the output accumulators.  pbase: slot-row index of the
// expert's first row in the activation chunk (act row r at chunk index
// pbase + r).
template <int BITS, int NR>
__device__ void down_stage(const Sh &sh, const uint8_t *stage, int rs, int cnt, int rowb, int K, uint32_t mask,
                           int pbase, const float *wgt)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int LPR = lanes_per_row(K), RPP = 32 / LPR, nsg = K / kSub;
    int rows[NR], nvalid;
    rows_from_mask<NR>(mask, rows, nvalid);
    int xoff[NR], soff[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int p = pbase + (r < nvalid ? r : nvalid - 1);
        xoff[r] = p * (K / 4);
        soff[r] = p * nsg;
    }
    const float4 *xs4 = reinterpret_cast<const float4 *>(sh.xs);
    const int first = rs + ((warp - rs % NCW) % NCW + NCW) % NCW;
    const int end = rs + cnt;
    const int n_owned = first < end ? (end - 1 - first) / NCW + 1 : 0;
    for (int i0 = 0; i0 < n_owned; i0 += RPP) {
        const int i = i0 + lane / LPR;
        const bool valid = i < n_owned;
        const int hl = first + i * NCW;
        float acc[1][NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[0][r] = 0.f;
        if (valid) {
            const uint8_t *const wr[1] = {stage + (size_t)(hl - rs) * rowb};
            for (int sg = lane % LPR; sg < nsg; sg += LPR)
                qdot_sub<BITS, NR, 1>(wr, K, sg, xs4, sh.xsum, xoff, soff, LPR, acc);
        }
        for (int o = LPR / 2; o >= 1; o >>= 1)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[0][r] += __shfl_xor_sync(FULLMASK, acc[0][r], o);
        if (valid && lane % LPR == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
                if (r < nvalid) sh.acc[hl * kMaxRows + rows[r]] += wgt[rows[r]] * acc[0][r];
        }
    }
}

__device__ __forceinline__ int nr_bucket(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

#define MOE_CASE(BV, RV, CALL) \
    case (BV) * 16 + (RV): { constexpr int B_ = (BV), R_ = (RV); CALL; } break;
#define MOE_CASES_NR(BV, CALL) MOE_CASE(BV, 1, CALL) MOE_CASE(BV, 2, CALL) MOE_CASE(BV, 4, CALL) MOE_CASE(BV, 8, CALL)

// Expert matrices: 4, 6 or 8 bits.
#define MOE_DISPATCH(BITSV, NRV, CALL)                                            \
    do {                                                                          \
        switch ((BITSV) * 16 + (NRV)) {                                           \
            MOE_CASES_NR(4, CALL) MOE_CASES_NR(6, CALL) MOE_CASES_NR(8, CALL)     \
        default: break;                                                           \
        }                                                                         \
    } while (0)

// Router rows: fp32 (0) or 4, 6, 8 bits.
#define MOE_DISPATCH_ROUTER(BITSV, NRV, CALL)                                                       \
    do {                                                                                            \
        switch ((BITSV) * 16 + (NRV)) {                                                             \
            MOE_CASES_NR(0, CALL) MOE_CASES_NR(4, CALL) MOE_CASES_NR(6, CALL) MOE_CASES_NR(8, CALL) \
        default: break;                                                                             \
        }                                                                                           \
    } while (0)

// ------------------------------------------------------------ P0: RMSNorm

// 1 / sqrt(mean(x^2) + eps) for the M bf16 rows of x (global) -> red[NCW*kMaxRows + m].
__device__ void row_rinv(const KParams &kp, const Sh &sh, const uint16_t *x)
{
    const int H = kp.g.H, M = kp.M, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float ss[kMaxRows];
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) ss[m] = 0.f;
    for (int j = tid * 8; j < H; j += NCT * 8) {
#pragma unroll
        for (int m = 0; m < kMaxRows; ++m) {
            if (m < M) {
                const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(x + (size_t)m * H + j));
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float a = __uint_as_float(wv[i] << 16), b = __uint_as_float(wv[i] & 0xFFFF0000u);
                    ss[m] = fmaf(a, a, ss[m]);
                    ss[m] = fmaf(b, b, ss[m]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) {
        const float t = warp_sum(ss[m]);
        if (lane == 0) sh.red[warp * kMaxRows + m] = t;
    }
    cbar();
    if (tid < M) {
        float t = 0.f;
        for (int w = 0; w < NCW; ++w) t += sh.red[w * kMaxRows + tid];
        sh.red[NCW * kMaxRows + tid] = rsqrtf(t / (float)H + kp.g.eps);
    }
    cbar();
}

// hn = x * rinv * gamma, arranged, with per-16 sums.
__device__ void build_hn(const KParams &kp, const Sh &sh, const uint16_t *x, const uint16_t *gamma)
{
    const int H = kp.g.H, M = kp.M, tid = threadIdx.x;
    row_rinv(kp, sh, x);
    const int nsg = H / kSub, LPR = lanes_per_row(H);
    for (int t = tid; t < M * nsg; t += NCT) {
        const int m = t / nsg, sg = t % nsg;
        const float rinv = sh.red[NCW * kMaxRows + m];
        const uint4 *xv = reinterpret_cast<const uint4 *>(x + (size_t)m * H + sg * 16);
        const uint4 *gv = reinterpret_cast<const uint4 *>(gamma + sg * 16);
        float v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 a = __ldcg(xv + h), g = __ldg(gv + h);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[h * 8 + 2 * i] = __uint_as_float(aw[i] << 16) * rinv * __uint_as_float(gw[i] << 16);
                v[h * 8 + 2 * i + 1] = __uint_as_float(aw[i] & 0xFFFF0000u) * rinv * __uint_as_float(gw[i] & 0xFFFF0000u);
            }
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) s += v[i];
        sh.xsum[m * nsg + sg] = s;
        float4 *xs4 = reinterpret_cast<float4 *>(sh.xs + (size_t)m * H);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            xs4[arr_index(sg, q, LPR)] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    cbar();
}

// ------------------------------------------------------------- R: routing

// Top-k of one row by a warp: threshold = k-th largest of the 32 lane
// maxima (a lower bound of the k-th largest overall), then exact ranks of
// the candidates above it.  Order: logit descending, expert id ascending.
__device__ void topk_row(const KParams &kp, const Sh &sh, int m, const float *logits)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = kp.g.E, k = kp.g.k, Er = kp.g.Er;
    constexpr int NPL = kMaxE / 32;
    float v[NPL];
    float bv = -FLT_MAX;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcg(logits + (size_t)m * Er + e) : -FLT_MAX;
        if (e < E && (v[i] > bv || (v[i] == bv && e < be))) { bv = v[i]; be = e; }
    }
    int rank = 0;
#pragma unroll 8
    for (int l = 0; l < 32; ++l) {
        const float ov = __shfl_sync(FULLMASK, bv, l);
        const int oe = __shfl_sync(FULLMASK, be, l);
        rank += (ov > bv || (ov == bv && oe < be)) ? 1 : 0;
    }
    const unsigned who = __ballot_sync(FULLMASK, rank == k - 1);
    const int src = __ffs(who) - 1;
    const float Tv = __shfl_sync(FULLMASK, bv, src);
    const int Te = __shfl_sync(FULLMASK, be, src);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && (v[i] > Tv || (v[i] == Tv && e <= Te))) ++cnt;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(FULLMASK, incl, o);
        if (lane >= o) incl += t;
    }
    const int C = __shfl_sync(FULLMASK, incl, 31);
    float *topv = sh.topv + m * kMaxK;
    int *tope = sh.tope + m * kMaxK;
    if (C <= kCandCap) {
        float *cv = sh.cand_v + warp * kCandCap;
        int *ce = sh.cand_e + warp * kCandCap;
        int pos = incl - cnt;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && (v[i] > Tv || (v[i] == Tv && e <= Te))) { cv[pos] = v[i]; ce[pos] = e; ++pos; }
        }
        __syncwarp();
        for (int c = lane; c < C; c += 32) {
            const float a = cv[c];
            const int ea = ce[c];
            int r = 0;
            for (int c2 = 0; c2 < C; ++c2) {
                const float b = cv[c2];
                r += (b > a || (b == a && ce[c2] < ea)) ? 1 : 0;
            }
            if (r < k) { topv[r] = a; tope[r] = ea; }
        }
    } else {
        // exact fallback: k rounds of warp arg-max
        unsigned taken = 0;
        for (int r = 0; r < k; ++r) {
            float lv = -FLT_MAX;
            int le = 0x7fffffff, li = -1;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !(taken >> i & 1u) && (v[i] > lv || (v[i] == lv && e < le))) { lv = v[i]; le = e; li = i; }
            }
            float gv = lv;
            int ge = le;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(FULLMASK, gv, o);
                const int oe = __shfl_xor_sync(FULLMASK, ge, o);
                if (ov > gv || (ov == gv && oe < ge)) { gv = ov; ge = oe; }
            }
            if (ge == le && li >= 0) taken |= 1u << li;
            if (lane == 0) { topv[r] = gv; tope[r] = ge; }
        }
    }
    __syncwarp();
    // renormalised softmax weights over the k kept logits (equal to the full
    // softmax probabilities divided by their top-k sum)
    float ev = 0.f;
    if (lane < k) ev = expf(topv[lane] - topv[0]);
    const float z = warp_sum(ev);
    if (lane < k) sh.topw[m * kMaxK + lane] = ev / z;
    if (lane == 0) {
        float sg = 0.f;
        if (kp.g.has_shared) {
            const float l = __ldcg(logits + (size_t)m * Er + E);
            sg = 1.0f / (1.0f + expf(-l));
        }
        sh.sigma[m] = sg;
    }
}

__device__ void route(const KParams &kp, const Sh &sh, const float *logits)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = kp.g.E, k = kp.g.k, M = kp.M;
    if (warp < M) topk_row(kp, sh, warp, logits);
    cbar();
    if (warp == 0) {
        for (int e = lane; e < E; e += 32) sh.emask[e] = 0u;
        __syncwarp();
        for (int t = lane; t < M * k; t += 32) atomicOr(&sh.emask[sh.tope[(t / k) * kMaxK + t % k]], 1u << (t / k));
        __syncwarp();
        int base = 0, rowbase = 0;
        for (int c0 = 0; c0 < E; c0 += 32) {
            const int e = c0 + lane;
            const uint32_t mk = e < E ? sh.emask[e] : 0u;
            const unsigned bal = __ballot_sync(FULLMASK, mk != 0u);
            const int pos = base + __popc(bal & ((1u << lane) - 1u));
            const int pc = mk ? __popc(mk) : 0;
            int inc = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULLMASK, inc, o);
                if (lane >= o) inc += t;
            }
            if (mk) {
                sh.slot_e[pos] = e;
                sh.slot_mask[pos] = mk;
                sh.eslot[e] = pos;
                const int rb0 = rowbase + inc - pc;
                sh.slot_rowbase[pos] = rb0;
                uint32_t mm = mk;
                for (int r = 0; mm; ++r) {
                    const int row = __ffs(mm) - 1;
                    mm &= mm - 1;
                    sh.pair_slot[rb0 + r] = pos;
                    sh.pair_m[rb0 + r] = row;
                }
            }
            base += __popc(bal);
            rowbase += __shfl_sync(FULLMASK, inc, 31);
        }
        if (lane == 0) {
            sh.flags[1] = base;
            sh.slot_rowbase[base] = rowbase;
        }
        __syncwarp();
        for (int t = lane; t < M * k; t += 32) {
            const int m = t / k, i = t % k;
            const int e = sh.tope[m * kMaxK + i];
            sh.slot_w[sh.eslot[e] * kMaxRows + m] = sh.topw[m * kMaxK + i];
            if (kp.mode == kModeRouter && blockIdx.x == 0) {
                kp.idx_out[m * k + i] = e;
                kp.w_out[m * k + i] = sh.topw[m * kMaxK + i];
            }
        }
    }
    cbar();
}

// ---------------------------------------------------------- workspace views

struct Ws {
    float *logits;   // [maxr][Er]
    float *act;      // [max_slots][maxr][I]
    float *act_s;    // [maxr][Is]
    uint16_t *ping[2];
};

__device__ __forceinline__ Ws ws_views(const KParams &kp)
{
    Ws w;
    w.logits = reinterpret_cast<float *>(kp.ws + kp.ws_l.off_logits);
    w.act = reinterpret_cast<float *>(kp.ws + kp.ws_l.off_act);
    w.act_s = reinterpret_cast<float *>(kp.ws + kp.ws_l.off_act_s);
    w.ping[0] = reinterpret_cast<uint16_t *>(kp.ws + kp.ws_l.off_ping);
    w.ping[1] = w.ping[0] + (size_t)kp.ws_l.maxr * kp.g.H;
    return w;
}

// ------------------------------------------------------------- the stages

// Stage schedule shared by the producer and the compute warps.  `f` gets
// (src, bytes, kind, slot, first, count) for each stage in order.
enum Kind { kRouter = 0, kSharedGU = 1, kGU = 2, kDown = 3, kSharedDown = 4 };

template <typename F>
__device__ __forceinline__ void phase1_stages(const KParams &kp, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    const int P = gridDim.x, c = blockIdx.x, S = kp.p.S;
    int a, b;
    split(g.Er, P, c, a, b);
    const int cr = S / g.rr_bytes;
    for (int r = a; r < b; r += cr) {
        const int n = min(cr, b - r);
        f(Lp.router + (size_t)r * g.rr_bytes, n * g.rr_bytes, kRouter, -1, r, n);
    }
    if (kp.mode == kModeLayers && g.has_shared) {
        split(g.Is, P, c, a, b);
        const int ub = 2 * g.sg_bytes, cu = S / ub;
        for (int j = a; j < b; j += cu) {
            const int n = min(cu, b - j);
            f(Lp.sgu + (size_t)j * ub, n * ub, kSharedGU, -1, j, n);
        }
    }
}

template <typename F>
__device__ __forceinline__ void phase2_stages(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    const int P = gridDim.x, c = blockIdx.x, S = kp.p.S;
    const int U = sh.flags[1];
    const int ub = 2 * g.g_bytes, cu = S / ub;
    int a, b;
    split(U * g.I, P, c, a, b);
    for (int n = a; n < b;) {
        const int s = n / g.I, j = n % g.I;
        const int cnt = min(cu, min(b, (s + 1) * g.I) - n);
        const int e = sh.slot_e[s];
        f(Lp.gu + ((size_t)e * g.I + j) * ub, cnt * ub, kGU, s, j, cnt);
        n += cnt;
    }
}

// Down stages of routed slots [s0, s1) (and of the shared expert when shared).
template <typename F>
__device__ __forceinline__ void down_stages(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, int s0, int s1,
                                            bool shared, F &&f)
{
    const Geo &g = kp.g;
    const int P = gridDim.x, c = blockIdx.x, S = kp.p.S;
    int h0, h1;
    split(g.H, P, c, h0, h1);
    const int nh = h1 - h0;
    if (!shared) {
        const int cd = S / g.d_bytes;
        for (int s = s0; s < s1; ++s) {
            const int e = sh.slot_e[s];
            for (int r = 0; r < nh; r += cd) {
                const int n = min(cd, nh - r);
                f(Lp.down + ((size_t)e * g.H + h0 + r) * g.d_bytes, n * g.d_bytes, kDown, s, r, n);
            }
        }
    } else {
        const int cd = S / g.sd_bytes;
        for (int r = 0; r < nh; r += cd) {
            const int n = min(cd, nh - r);
            f(Lp.sdown + (size_t)(h0 + r) * g.sd_bytes, n * g.sd_bytes, kSharedDown, -1, r, n);
        }
    }
}

// Routed slots of P3 are processed in chunks whose activations fit in xs.
__device__ __forceinline__ int chunk_end(const KParams &kp, const Sh &sh, int s, int U)
{
    const int cap = (kp.p.maxr * kp.g.H) / kp.g.I;
    const int base = sh.slot_rowbase[s];
    int se = s + 1;
    while (se < U && sh.slot_rowbase[se + 1] - base <= cap) ++se;
    return se;
}

// ------------------------------------------------------------- producer

__device__ bool issue(const Sh &sh, unsigned &q, const uint8_t *src, int bytes)
{
    const int slot = (int)(q % (unsigned)sh.NS);
    const unsigned n = q / (unsigned)sh.NS;
    if (n > 0 && !wait_bar(sh, &sh.empty[slot], (n - 1) & 1u, 1)) return false;
    if (aborted(sh)) return false;
    mbar_expect_tx(&sh.full[slot], (unsigned)bytes);
    bulk_load(sh.ring + (size_t)slot * sh.S, src, (unsigned)bytes, &sh.full[slot]);
    ++q;
    return true;
}

__device__ void producer(const KParams &kp, const Sh &sh)
{
    unsigned q = 0;
    bool ok = true;
    for (int l = 0; l < kp.L && ok; ++l) {
        const LayerPtrs &Lp = kp.layer[l];
        phase1_stages(kp, Lp, [&](const uint8_t *src, int bytes, int, int, int, int) {
            if (ok) ok = issue(sh, q, src, bytes);
        });
        if (!ok || kp.mode == kModeRouter) break;
        if (!wait_bar(sh, sh.route, (unsigned)l & 1u, 2)) break;
        phase2_stages(kp, sh, Lp, [&](const uint8_t *src, int bytes, int, int, int, int) {
            if (ok) ok = issue(sh, q, src, bytes);
        });
        const int U = sh.flags[1];
        down_stages(kp, sh, Lp, 0, U, false, [&](const uint8_t *src, int bytes, int, int, int, int) {
            if (ok) ok = issue(sh, q, src, bytes);
        });
        if (kp.g.has_shared)
            down_stages(kp, sh, Lp, 0, 0, true, [&](const uint8_t *src, int bytes, int, int, int, int) {
                if (ok) ok = issue(sh, q, src, bytes);
            });
    }
    // Let every copy still in flight land before the CTA can exit.
    const unsigned first = q > (unsigned)sh.NS ? q - (unsigned)sh.NS : 0u;
    for (unsigned t = first; t < q; ++t) {
        const int slot = (int)(t % (unsigned)sh.NS);
        const unsigned long long t0 = now_ns();
        while (!mbar_try_wait(&sh.full[slot], (t / (unsigned)sh.NS) & 1u))
            if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) break;
    }
}

// -------------------------------------------------------- compute warps

__device__ __forceinline__ const uint8_t *stage_ptr(const Sh &sh, unsigned q)
{
    return sh.ring + (size_t)(q % (unsigned)sh.NS) * sh.S;
}

__device__ __forceinline__ bool stage_wait(const Sh &sh, unsigned q, int where)
{
    return wait_bar(sh, &sh.full[q % (unsigned)sh.NS], (q / (unsigned)sh.NS) & 1u, where);
}

// single-consumer release: the whole arrival count at once
__device__ __forceinline__ void stage_release_all(const Sh &sh, unsigned q)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[q % (unsigned)sh.NS], NCW);
}

__device__ __forceinline__ void stage_release_one(const Sh &sh, unsigned q)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[q % (unsigned)sh.NS], 1);
}

__device__ void phase1(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w)
{
    const int warp = threadIdx.x >> 5;
    const Geo &g = kp.g;
    const uint32_t all = (1u << kp.M) - 1u;
    const int nr = nr_bucket(kp.M);
    phase1_stages(kp, Lp, [&](const uint8_t *, int, int kind, int, int first, int n) {
        const unsigned me = q++;
        if ((int)(me % NCW) != warp) return;
        if (!aborted(sh) && stage_wait(sh, me, 10)) {
            const uint8_t *st = stage_ptr(sh, me);
            if (kind == kRouter) {
                MOE_DISPATCH_ROUTER(g.qb, nr, (router_stage<B_, R_>(sh, st, n, g.rr_bytes, g.H, all, w.logits, g.Er, first)));
            } else {
                MOE_DISPATCH(g.sb, nr, (gu_stage<B_, R_>(sh, st, n, g.sg_bytes, g.H, all, w.act_s, g.Is, first)));
            }
        }
        stage_release_all(sh, me);
    });
}

__device__ void phase2(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w)
{
    const int warp = threadIdx.x >> 5;
    const Geo &g = kp.g;
    const int maxr = kp.ws_l.maxr;
    phase2_stages(kp, sh, Lp, [&](const uint8_t *, int, int, int s, int first, int n) {
        const unsigned me = q++;
        if ((int)(me % NCW) != warp) return;
        if (!aborted(sh) && stage_wait(sh, me, 20)) {
            const uint32_t mask = sh.slot_mask[s];
            const int nr = nr_bucket(__popc(mask));
            float *act = w.act + (size_t)s * maxr * g.I;
            MOE_DISPATCH(g.rb, nr, (gu_stage<B_, R_>(sh, stage_ptr(sh, me), n, g.g_bytes, g.H, mask, act, g.I, first)));
        }
        stage_release_all(sh, me);
    });
}

// Load activation rows (pairs [p0, p1) of the slot-row list, or the shared
// expert's M rows) into xs/xsum in the arranged layout.
__device__ void load_act(const KParams &kp, const Sh &sh, const Ws &w, int p0, int p1, bool shared)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = kp.g;
    const int K = shared ? g.Is : g.I;
    const int LPR = lanes_per_row(K), nsg = K / kSub, nf = K / 4;
    const int maxr = kp.ws_l.maxr;
    const int npairs = shared ? kp.M : p1 - p0;
    for (int pi = warp; pi < npairs; pi += NCW) {
        const float *src;
        if (shared) {
            src = w.act_s + (size_t)pi * g.Is;
        } else {
            const int p = p0 + pi;
            src = w.act + ((size_t)sh.pair_slot[p] * maxr + sh.pair_m[p]) * g.I;
        }
        float4 *dst = reinterpret_cast<float4 *>(sh.xs) + (size_t)pi * nf;
        float *dsum = sh.xsum + (size_t)pi * nsg;
        for (int f0 = 0; f0 < nf; f0 += 32) {
            const int f = f0 + lane;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (f < nf) v = __ldcg(reinterpret_cast<const float4 *>(src) + f);
            float s = (v.x + v.y) + (v.z + v.w);
            s += __shfl_xor_sync(FULLMASK, s, 1);
            s += __shfl_xor_sync(FULLMASK, s, 2);
            if (f < nf) {
                const int sg = f >> 2, t = f & 3;
                dst[arr_index(sg, t, LPR)] = v;
                if (t == 0) dsum[sg] = s;
            }
        }
    }
}

__device__ bool phase3(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w,
                       const uint16_t *xin, uint16_t *xout)
{
    const Geo &g = kp.g;
    const int tid = threadIdx.x, P = gridDim.x, c = blockIdx.x;
    int h0, h1;
    split(g.H, P, c, h0, h1);
    const int nh = h1 - h0;
    for (int t = tid; t < nh * kMaxRows; t += NCT) sh.acc[t] = 0.f;
    const int U = sh.flags[1];
    for (int s = 0; s < U;) {
        const int se = chunk_end(kp, sh, s, U);
        if (cbar_or(aborted(sh))) return false;
        const int p0 = sh.slot_rowbase[s];
        load_act(kp, sh, w, p0, sh.slot_rowbase[se], false);
        if (cbar_or(aborted(sh))) return false;
        down_stages(kp, sh, Lp, s, se, false, [&](const uint8_t *, int, int, int slot, int first, int n) {
            const unsigned me = q++;
            if (!aborted(sh) && stage_wait(sh, me, 30)) {
                const uint32_t mask = sh.slot_mask[slot];
                const int nr = nr_bucket(__popc(mask));
                MOE_DISPATCH(g.rb, nr, (down_stage<B_, R_>(sh, stage_ptr(sh, me), first, n, g.d_bytes, g.I, mask,
                                                          sh.slot_rowbase[slot] - p0, sh.slot_w + slot * kMaxRows)));
            }
            stage_release_one(sh, me);
        });
        s = se;
    }
    if (g.has_shared) {
        if (cbar_or(aborted(sh))) return false;
        load_act(kp, sh, w, 0, 0, true);
        if (cbar_or(aborted(sh))) return false;
        const uint32_t all = (1u << kp.M) - 1u;
        const int nr = nr_bucket(kp.M);
        down_stages(kp, sh, Lp, 0, 0, true, [&](const uint8_t *, int, int, int, int first, int n) {
            const unsigned me = q++;
            if (!aborted(sh) && stage_wait(sh, me, 40)) {
                MOE_DISPATCH(g.sb, nr, (down_stage<B_, R_>(sh, stage_ptr(sh, me), first, n, g.sd_bytes, g.Is, all, 0,
                                                          sh.sigma)));
            }
            stage_release_one(sh, me);
        });
    }
    if (cbar_or(aborted(sh))) return false;
    // residual + bf16 rounding of this CTA's outputs
    const int M = kp.M;
    for (int t = tid; t < nh * M; t += NCT) {
        const int hl = t / M, m = t % M;
        const size_t idx = (size_t)m * g.H + h0 + hl;
        const float o = bf2f(__ldcg(xin + idx)) + sh.acc[hl * kMaxRows + m];
        xout[idx] = f2bf(o);
    }
    return true;
}

// out_n = bf16(out * rinv * gamma_next) for this CTA's outputs.
__device__ void write_normed(const KParams &kp, const Sh &sh, const uint16_t *out, const uint16_t *gamma_next)
{
    const Geo &g = kp.g;
    row_rinv(kp, sh, out);
    int h0, h1;
    split(g.H, gridDim.x, blockIdx.x, h0, h1);
    const int nh = h1 - h0, M = kp.M;
    for (int t = threadIdx.x; t < nh * M; t += NCT) {
        const int hl = t / M, m = t % M;
        const size_t idx = (size_t)m * g.H + h0 + hl;
        const float v = bf2f(__ldcg(out + idx)) * sh.red[NCW * kMaxRows + m] * bf2f(gamma_next[h0 + hl]);
        kp.out_normed[idx] = f2bf(v);
    }
}

__device__ void compute(const KParams &kp, const Sh &sh)
{
    const Ws w = ws_views(kp);
    unsigned q = 0;
    unsigned gen = 0;
    int nsync = 0;
    if (threadIdx.x == 0) gen = *(volatile unsigned *)&sh.ctrl->gen;
    for (int l = 0; l < kp.L; ++l) {
        const LayerPtrs &Lp = kp.layer[l];
        const bool last = l == kp.L - 1;
        const uint16_t *xin = l == 0 ? kp.x : w.ping[(l - 1) & 1];
        uint16_t *xout = last ? kp.out : w.ping[l & 1];
        build_hn(kp, sh, xin, Lp.gamma);
        phase1(kp, sh, Lp, q, w);
        if (!grid_sync(kp, sh, gen, nsync)) return;
        route(kp, sh, w.logits);
        if (kp.mode == kModeRouter) return;
        if (threadIdx.x == 0) mbar_arrive(sh.route, 1);
        phase2(kp, sh, Lp, q, w);
        if (!grid_sync(kp, sh, gen, nsync)) return;
        if (!phase3(kp, sh, Lp, q, w, xin, xout)) return;
        if (!last || kp.out_normed) {
            if (!grid_sync(kp, sh, gen, nsync)) return;
        }
        if (last && kp.out_normed) write_normed(kp, sh, xout, Lp.gamma_next);
    }
}

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ KParams kp)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = carve(kp.g, kp.p);
    Sh sh;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar);
    sh.full = bars;
    sh.empty = bars + kp.p.NS;
    sh.route = bars + 2 * kp.p.NS;
    sh.flags = reinterpret_cast<int *>(smem + L.flags);
    sh.slot_e = reinterpret_cast<int *>(smem + L.slot_e);
    sh.slot_mask = reinterpret_cast<uint32_t *>(smem + L.slot_mask);
    sh.slot_rowbase = reinterpret_cast<int *>(smem + L.slot_rowbase);
    sh.slot_w = reinterpret_cast<float *>(smem + L.slot_w);
    sh.sigma = reinterpret_cast<float *>(smem + L.sigma);
    sh.eslot = reinterpret_cast<int *>(smem + L.eslot);
    sh.emask = reinterpret_cast<uint32_t *>(smem + L.emask);
    sh.topv = reinterpret_cast<float *>(smem + L.topv);
    sh.tope = reinterpret_cast<int *>(smem + L.tope);
    sh.topw = reinterpret_cast<float *>(smem + L.topw);
    sh.cand_v = reinterpret_cast<float *>(smem + L.cand_v);
    sh.cand_e = reinterpret_cast<int *>(smem + L.cand_e);
    sh.pair_slot = reinterpret_cast<int *>(smem + L.pair_slot);
    sh.pair_m = reinterpret_cast<int *>(smem + L.pair_m);
    sh.red = reinterpret_cast<float *>(smem + L.red);
    sh.xs = reinterpret_cast<float *>(smem + L.xs);
    sh.xsum = reinterpret_cast<float *>(smem + L.xsum);
    sh.acc = reinterpret_cast<float *>(smem + L.acc);
    sh.ring = smem + L.ring;
    sh.NS = kp.p.NS;
    sh.S = kp.p.S;
    sh.timeout_ns = kp.timeout_ns;
    sh.ctrl = reinterpret_cast<Ctrl *>(kp.ws);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kp.p.NS; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], NCW);
        }
        mbar_init(sh.route, 1);
        sh.flags[0] = 0;
        sh.flags[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) producer(kp, sh);
        return;
    }
    compute(kp, sh);
}

int g_num_sms[64];
bool g_attr_set[64];

}  // namespace

bool make_plan(const Geo &g, int maxr, int num_sms, Plan &p)
{
    p.P = num_sms;
    p.maxr = maxr;
    p.max_slots = g.E < maxr * g.k ? g.E : maxr * g.k;
    p.hrows = (g.H + num_sms - 1) / num_sms + 1;
    const int unit = 2 * g.g_bytes;
    int maxi = g.rr_bytes;
    if (unit > maxi) maxi = unit;
    if (g.d_bytes > maxi) maxi = g.d_bytes;
    if (g.has_shared) {
        if (2 * g.sg_bytes > maxi) maxi = 2 * g.sg_bytes;
        if (g.sd_bytes > maxi) maxi = g.sd_bytes;
    }
    p.S = (maxi + unit - 1) / unit * unit;
    p.NS = 2;
    const int fixed = carve(g, p).ring;  // everything before the ring
    const int room = kSmemMax - fixed - 256;
    int ns = room / p.S;
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 2) return false;
    p.NS = ns;
    p.smem_bytes = carve(g, p).total;
    return p.smem_bytes <= kSmemMax;
}

int launch_decode(const KParams &kp, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    if (!g_attr_set[dev]) {
        e = cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
        g_attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)kp.p.P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)kp.p.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe_decode_kernel, kp);
    note_launch();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

int device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

}  // namespace moe
