// Persistent decode kernel of the quantized MoE FFN layer (and of a stack of
// such layers) for sm_103a.
//
// One CTA per SM: 16 compute warps and one producer warp.  Eight lanes of the
// producer warp stream every weight byte the CTA needs through a ring of
// shared-memory stages with 1-D bulk copies (cp.async.bulk completing on
// mbarrier transaction counts); several issuing lanes are needed because one
// thread cannot issue small bulk copies fast enough to fill HBM.  Each stage
// is consumed by one compute warp, which dequantises in registers and
// accumulates in fp32.  Per layer:
//
//   P0  every CTA: RMSNorm of the M input rows into shared memory
//       (flash-moe, "Metal Compute Shaders": RMS normalisation)
//   P1  router rows (plus the shared-expert gate row) and the shared
//       expert's gate/up units, split over the CTAs          -> grid barrier
//   R   every CTA: softmax + top-k + renormalisation per row and the list of
//       distinct selected experts with the rows that chose each
//       (PureDrive model card, "Summary": the full top-8 of 256 is kept)
//   P1b the shared expert's down rows of this CTA's output slice (weights
//       prefetched before routing is known)
//   P2  gate/up units of the selected experts, each expert streamed once for
//       all the rows that chose it (model card, "How it works": the verify
//       pass reads its weights once), SwiGLU                 -> grid barrier
//   P3  down rows of every selected expert for this CTA's output slice
//   C   weighted combine + sigmoid-gated shared expert + residual, bf16
//       (flash-moe: "MoE combine + residual + gate")         -> grid barrier
//   N   the fused next RMSNorm of the bf16 output (model card: fused
//       add+RMSNorm), or the next layer's P0.
//
// Determinism: no float atomics; every sum has a fixed order that depends
// only on the row itself, so row m of an M-row call equals a 1-row call.
#include <cuda_bf16.h>

#include <cfloat>
#include <type_traits>

#include "moe_internal.h"
#include "moe_unpack.cuh"

namespace moe {
namespace {

constexpr int NCW = kConsumerWarps;
constexpr int NCT = NCW * 32;
constexpr int NP = kProducerLanes;
constexpr int kCandCap = 64;
constexpr int kRedChunks = 8;        // per-row partial sums in the RMSNorm reduction
constexpr unsigned FULLMASK = 0xffffffffu;

// ------------------------------------------------------------ shared layout

struct SmemLayout {
    int bar, flags, slot_e, slot_mask, slot_rowbase, sigma, eslot, emask, topv, tope, topw;
    int row_w, row_pair, cand_v, cand_e, red, xs, xsum, ybuf, ysh, target, ring, total;
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
    L.sigma = take(o, kMaxRows * 4, 4);
    L.eslot = take(o, g.E * 4, 4);
    L.emask = take(o, g.E * 4, 4);
    L.topv = take(o, kMaxRows * kMaxK * 4, 4);
    L.tope = take(o, kMaxRows * kMaxK * 4, 4);
    L.topw = take(o, kMaxRows * kMaxK * 4, 4);
    L.row_w = take(o, kMaxRows * kMaxK * 4, 4);
    L.row_pair = take(o, kMaxRows * kMaxK * 4, 4);
    L.cand_v = take(o, kMaxRows * kCandCap * 4, 4);
    L.cand_e = take(o, kMaxRows * kCandCap * 4, 4);
    L.red = take(o, kMaxRows * (kRedChunks + 1) * 4, 4);
    L.xs = take(o, p.maxr * g.H * 4, 16);
    L.xsum = take(o, p.maxr * (g.H / kSub) * 4, 16);
    L.ybuf = take(o, p.maxr * g.k * p.hrows * 4, 16);
    L.ysh = take(o, p.hrows * kMaxRows * 4, 16);
    L.target = take(o, ms * 4, 16);
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

// The same, letting the hardware suspend the thread for up to `ns`
// nanoseconds while the phase is incomplete (waiting warps then take no
// issue slots from the computing ones).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, unsigned parity, unsigned ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(ns) : "memory");
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

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

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

// Phase stamp (thread 0 of the compute warps, or a producer lane).
__device__ __forceinline__ void stamp(const KParams &kp, int l, int ev)
{
    if (kp.trace && l < kMaxLayers)
        kp.trace[((size_t)blockIdx.x * kMaxLayers + l) * kTraceEvents + ev] = now_ns();
}

// Per-warp timeline (lane 0 of each compute warp) of CTAs 0 and gridDim/2,
// stored after the per-CTA stamps: [2][kMaxLayers][16 warps][16 events].
__device__ __forceinline__ void wstamp(const KParams &kp, int l, int ev)
{
    if (!kp.trace || l >= kMaxLayers || (threadIdx.x & 31) != 0) return;
    const int c = blockIdx.x == 0 ? 0 : (blockIdx.x == gridDim.x / 2 ? 1 : -1);
    if (c < 0) return;
    const size_t base = (size_t)gridDim.x * kMaxLayers * kTraceEvents;
    kp.trace[base + (((size_t)c * kMaxLayers + l) * 16 + (threadIdx.x >> 5)) * 16 + ev] = now_ns();
}

// ----------------------------------------------------------- CTA state

struct Sh {
    uint64_t *full, *empty, *route;
    int *flags;          // [0] abort, [1] U
    int *slot_e;
    uint32_t *slot_mask;
    int *slot_rowbase;
    float *sigma;        // [kMaxRows]
    int *eslot;
    uint32_t *emask;
    float *topv;         // [kMaxRows][kMaxK]  by weight
    int *tope;
    float *topw;
    float *row_w;        // [kMaxRows][kMaxK]  by expert id
    int *row_pair;
    float *cand_v;       // [kMaxRows][kCandCap]
    int *cand_e;
    float *red;          // [kMaxRows][kRedChunks + 1]
    float *xs;           // arranged hn rows
    float *xsum;         // per-16 sums of xs
    float *ybuf;         // [pair][hrows] routed expert outputs of this CTA's slice
    float *ysh;          // [hrows][kMaxRows] shared expert outputs
    unsigned *target;    // [max_slots] activation-ready count each slot must reach this layer
    unsigned *act_done;  // [max_slots] global activation-ready counters (workspace)
    uint8_t *ring;
    int NS, S, hrows;
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
        if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
        if ((it & 7) == 0) {
            if (aborted(sh)) return false;
            if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) {
                raise_abort(sh, where);
                return false;
            }
        }
    }
}

// Bounded wait (lane 0 polls, the warp follows) until a global counter
// reaches `target`; false on timeout or abort.
__device__ bool wait_count(const Sh &sh, const unsigned *ctr, unsigned target, int where)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0 && ld_acquire(ctr) < target) {
        const unsigned long long t0 = now_ns();
        for (unsigned it = 1;; ++it) {
            __nanosleep(64);   // many warps poll: keep the L2 traffic low
            if (ld_acquire(ctr) >= target) break;
            if ((it & 31) == 0) {
                if (aborted(sh)) { ok = false; break; }
                if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) { raise_abort(sh, where); ok = false; break; }
            }
        }
    }
    return __shfl_sync(FULLMASK, ok ? 1 : 0, 0) != 0;
}

// Grid-wide barrier over the compute warps of every CTA.  The arrival
// counter grows monotonically during a launch (barrier b waits for
// (b + 1) * gridDim.x arrivals) and is reset by the last CTA to finish.
__device__ bool grid_sync(const KParams &kp, const Sh &sh, int &nsync)
{
    if (cbar_or(aborted(sh))) return false;
    if (threadIdx.x == 0) {
        Ctrl *ctrl = sh.ctrl;
        const unsigned target = (unsigned)(nsync + 1) * gridDim.x;
        if (!(kp.skip_cta == (int)blockIdx.x && nsync == 0)) red_release_add(&ctrl->count, 1u);
        if (ld_acquire(&ctrl->count) < target) {
            const unsigned long long t0 = now_ns();
            for (unsigned it = 1;; ++it) {
                if (ld_acquire(&ctrl->count) >= target) break;
                if ((it & 63) == 0) {
                    if (*(volatile int *)&ctrl->status != 0) { *(volatile int *)&sh.flags[0] = 1; break; }
                    if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) { raise_abort(sh, 100 + nsync); break; }
                }
            }
        }
    }
    nsync += 1;
    return !cbar_or(aborted(sh));
}

__device__ void kernel_exit(const Sh &sh, int sh_max_slots_for_reset)
{
    if (threadIdx.x == 0 && !aborted(sh)) {
        Ctrl *ctrl = sh.ctrl;
        const unsigned old = atom_add_acqrel(&ctrl->exit, 1u);
        if (old == gridDim.x - 1) {
            for (int i = 0; i < sh_max_slots_for_reset; ++i) st_relaxed(&sh.act_done[i], 0u);
            st_relaxed(&ctrl->count, 0u);
            st_relaxed(&ctrl->exit, 0u);
        }
    }
}

__device__ __forceinline__ void split(int n, int P, int c, int &a, int &b)
{
    a = (int)((long long)n * c / P);
    b = (int)((long long)n * (c + 1) / P);
}

// ------------------------------------------------------ dot-product kernels

// Arranged float4 index of (sub-group sg, quarter t) for vectors of K inputs:
// lanes holding consecutive sub-groups read consecutive float4s.  LPR is a
// power of two (16-input sub-groups per row, capped at 32).
__device__ __forceinline__ int arr_index(int sg, int t, int LPR)
{
    return ((sg & ~(LPR - 1)) << 2) + t * LPR + (sg & (LPR - 1));
}

template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t *row, int sg, uint32_t (&w)[4])
{
    if (BITS == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + sg * 8);
        w[0] = v.x; w[1] = v.y; w[2] = 0; w[3] = 0;
    } else if (BITS == 6) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(row + sg * 12);
        w[0] = p[0]; w[1] = p[1]; w[2] = p[2]; w[3] = 0;
    } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + sg * 16);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
}

__device__ __forceinline__ void scale_bias(const uint8_t *row, int K, int bits, int sg, float &s, float &b)
{
    const uint32_t sbw = *reinterpret_cast<const uint32_t *>(row + K * bits / 8 + (sg >> 2) * 4);
    s = __uint_as_float(sbw << 16);
    b = __uint_as_float(sbw & 0xFFFF0000u);
}

// Codes 4T .. 4T+3 of NROWS weight rows as two exact float pairs per row
// (packed two-lane FADD removes the exponent offsets).
template <int BITS, int NROWS, int T>
__device__ __forceinline__ void codes4(const uint32_t (&w)[NROWS][4], float2 (&qa)[NROWS], float2 (&qb)[NROWS])
{
#pragma unroll
    for (int n = 0; n < NROWS; ++n) {
        float f[4], o[4];
        Unpack<BITS>::template raw4<T>(w[n], f, o);
        qa[n] = __fadd2_rn(make_float2(f[0], f[1]), make_float2(-o[0], -o[1]));
        qb[n] = __fadd2_rn(make_float2(f[2], f[3]), make_float2(-o[2], -o[3]));
    }
}

// Sub-group sg (16 inputs) of NROWS weight rows against NR activation rows
// arranged in shared memory: acc[n][r] += s_g * sum(q x) + b_g * sum(x), the
// per-group affine factoring of sum_j (q_j s + b) x_j.  Two-lane FMAs keep
// codes 0, 2 and 1, 3 of each quarter in separate partial sums.
template <int BITS, int NR, int NROWS, int T>
__device__ __forceinline__ void quarter_s(const uint32_t (&w)[NROWS][4], const float4 *xs4, const int (&xoff)[NR],
                                          int ai, int LPR, float2 (&S)[NROWS][NR])
{
    float2 qa[NROWS], qb[NROWS];
    codes4<BITS, NROWS, T>(w, qa, qb);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float4 x = xs4[xoff[r] + ai + T * LPR];
        const float2 xa = make_float2(x.x, x.y), xb = make_float2(x.z, x.w);
#pragma unroll
        for (int n = 0; n < NROWS; ++n) {
            S[n][r] = __ffma2_rn(qa[n], xa, S[n][r]);
            S[n][r] = __ffma2_rn(qb[n], xb, S[n][r]);
        }
    }
}

template <int BITS, int NR, int NROWS>
__device__ __forceinline__ void qdot_sub(const uint8_t *const (&wr)[NROWS], int K, int sg, const float4 *xs4,
                                         const float *xsum, const int (&xoff)[NR], const int (&soff)[NR],
                                         int LPR, float (&acc)[NROWS][NR])
{
    const int ai = arr_index(sg, 0, LPR);
    if constexpr (BITS == 0) {
#pragma unroll
        for (int n = 0; n < NROWS; ++n) {
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
    } else {
        uint32_t w[NROWS][4];
        float s[NROWS], b[NROWS];
#pragma unroll
        for (int n = 0; n < NROWS; ++n) {
            load_codes<BITS>(wr[n], sg, w[n]);
            scale_bias(wr[n], K, BITS, sg, s[n], b[n]);
        }
        float2 S[NROWS][NR];
#pragma unroll
        for (int n = 0; n < NROWS; ++n)
#pragma unroll
            for (int r = 0; r < NR; ++r) S[n][r] = make_float2(0.f, 0.f);
        quarter_s<BITS, NR, NROWS, 0>(w, xs4, xoff, ai, LPR, S);
        quarter_s<BITS, NR, NROWS, 1>(w, xs4, xoff, ai, LPR, S);
        quarter_s<BITS, NR, NROWS, 2>(w, xs4, xoff, ai, LPR, S);
        quarter_s<BITS, NR, NROWS, 3>(w, xs4, xoff, ai, LPR, S);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float xsm = xsum[soff[r] + sg];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) {
                acc[n][r] = fmaf(s[n], S[n][r].x + S[n][r].y, acc[n][r]);
                acc[n][r] = fmaf(b[n], xsm, acc[n][r]);
            }
        }
    }
}

// The same against NR activation rows held in registers (16 values of the
// lane's sub-group and their sum per row).
template <int BITS, int NR, int NROWS>
__device__ __forceinline__ void rdot_sub(const uint8_t *const (&wr)[NROWS], int K, int sg, const float (&a)[NR][16],
                                         const float (&as)[NR], float (&acc)[NROWS][NR])
{
    uint32_t w[NROWS][4];
    float s[NROWS], b[NROWS];
#pragma unroll
    for (int n = 0; n < NROWS; ++n) {
        load_codes<BITS>(wr[n], sg, w[n]);
        scale_bias(wr[n], K, BITS, sg, s[n], b[n]);
    }
    float2 S[NROWS][NR];
#pragma unroll
    for (int n = 0; n < NROWS; ++n)
#pragma unroll
        for (int r = 0; r < NR; ++r) S[n][r] = make_float2(0.f, 0.f);
    float2 qa[NROWS], qb[NROWS];
#define MOE_RQ(T)                                                                                 \
    codes4<BITS, NROWS, T>(w, qa, qb);                                                            \
    _Pragma("unroll") for (int r = 0; r < NR; ++r) {                                              \
        const float2 xa = make_float2(a[r][4 * T], a[r][4 * T + 1]);                              \
        const float2 xb = make_float2(a[r][4 * T + 2], a[r][4 * T + 3]);                          \
        _Pragma("unroll") for (int n = 0; n < NROWS; ++n) {                                       \
            S[n][r] = __ffma2_rn(qa[n], xa, S[n][r]);                                             \
            S[n][r] = __ffma2_rn(qb[n], xb, S[n][r]);                                             \
        }                                                                                         \
    }
    MOE_RQ(0) MOE_RQ(1) MOE_RQ(2) MOE_RQ(3)
#undef MOE_RQ
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int n = 0; n < NROWS; ++n) {
            acc[n][r] = fmaf(s[n], S[n][r].x + S[n][r].y, acc[n][r]);
            acc[n][r] = fmaf(b[n], as[r], acc[n][r]);
        }
}

// Token rows first .. first + NR - 1 of a row mask (in set-bit order),
// padded with the last one.
template <int NR>
__device__ __forceinline__ void rows_of_group(uint32_t mask, int first, int (&rows)[NR], int &nvalid)
{
    for (int i = 0; i < first; ++i) mask &= mask - 1;
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

__device__ __forceinline__ int nr_bucket(int n) { return n <= 1 ? 1 : 2; }

template <int N, int NR>
__device__ __forceinline__ void lane_reduce(float (&acc)[N][NR], int LPR)
{
    for (int o = LPR / 2; o >= 1; o >>= 1)
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[n][r] += __shfl_xor_sync(FULLMASK, acc[n][r], o);
}

// Gate/up units (gate row, up row) of one stage for NR token rows of hn, NU
// units per lane group at a time -> act[m * mstride + j0 + u] = silu(g) * up.
template <int BITS, int NR, int NU>
__device__ void gu_pass(const Sh &sh, const uint8_t *stage, int cnt, int rowb, int H, const int (&rows)[NR],
                        int nvalid, float *act, int mstride, int j0)
{
    const int lane = threadIdx.x & 31;
    const int LPR = lanes_per_row(H), RPP = 32 / LPR, nsg = H / kSub;
    int xoff[NR], soff[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) { xoff[r] = rows[r] * (H / 4); soff[r] = rows[r] * nsg; }
    const float4 *xs4 = reinterpret_cast<const float4 *>(sh.xs);
    for (int u0 = 0; u0 < cnt; u0 += RPP * NU) {
        const int ub = u0 + (lane / LPR) * NU;
        const uint8_t *wr[2 * NU];
#pragma unroll
        for (int i = 0; i < NU; ++i) {
            const int u = ub + i < cnt ? ub + i : 0;
            wr[2 * i] = stage + (size_t)u * 2 * rowb;
            wr[2 * i + 1] = wr[2 * i] + rowb;
        }
        float acc[2 * NU][NR];
#pragma unroll
        for (int n = 0; n < 2 * NU; ++n)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[n][r] = 0.f;
        if (ub < cnt)
            for (int sg = lane % LPR; sg < nsg; sg += LPR)
                qdot_sub<BITS, NR, 2 * NU>(wr, H, sg, xs4, sh.xsum, xoff, soff, LPR, acc);
        lane_reduce<2 * NU, NR>(acc, LPR);
        if (lane % LPR == 0) {
#pragma unroll
            for (int i = 0; i < NU; ++i)
                if (ub + i < cnt) {
#pragma unroll
                    for (int r = 0; r < NR; ++r)
                        if (r < nvalid) {
                            const float g = acc[2 * i][r], up = acc[2 * i + 1][r];
                            act[(size_t)rows[r] * mstride + j0 + ub + i] = g / (1.0f + expf(-g)) * up;
                        }
                }
        }
    }
}

// Router rows of one stage, NU rows per lane group at a time -> logits[m * Er + e0 + u].
template <int BITS, int NR, int NU>
__device__ void router_pass(const Sh &sh, const uint8_t *stage, int cnt, int rowb, int H, const int (&rows)[NR],
                            int nvalid, float *logits, int Er, int e0)
{
    const int lane = threadIdx.x & 31;
    const int LPR = lanes_per_row(H), RPP = 32 / LPR, nsg = H / kSub;
    int xoff[NR], soff[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) { xoff[r] = rows[r] * (H / 4); soff[r] = rows[r] * nsg; }
    const float4 *xs4 = reinterpret_cast<const float4 *>(sh.xs);
    for (int u0 = 0; u0 < cnt; u0 += RPP * NU) {
        const int ub = u0 + (lane / LPR) * NU;
        const uint8_t *wr[NU];
#pragma unroll
        for (int i = 0; i < NU; ++i) wr[i] = stage + (size_t)(ub + i < cnt ? ub + i : 0) * rowb;
        float acc[NU][NR];
#pragma unroll
        for (int n = 0; n < NU; ++n)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[n][r] = 0.f;
        if (ub < cnt)
            for (int sg = lane % LPR; sg < nsg; sg += LPR)
                qdot_sub<BITS, NR, NU>(wr, H, sg, xs4, sh.xsum, xoff, soff, LPR, acc);
        lane_reduce<NU, NR>(acc, LPR);
        if (lane % LPR == 0) {
#pragma unroll
            for (int i = 0; i < NU; ++i)
                if (ub + i < cnt) {
#pragma unroll
                    for (int r = 0; r < NR; ++r)
                        if (r < nvalid) logits[(size_t)rows[r] * Er + e0 + ub + i] = acc[i][r];
                }
        }
    }
}

// Down rows [rs, rs + cnt) (relative to the CTA's first output) of one
// expert for NR token rows whose activations (K inputs each) the warp keeps
// in registers: lane l holds sub-groups l mod LPR (+ LPR * i, i < SPL); NU
// rows per lane group at a time.  Output of token row r, row h:
// y[yoff[r] + h * ystride].
template <int BITS, int NR, int SPL, int NU>
__device__ void dn_pass(const uint8_t *stage, int rs, int cnt, int rowb, int K, const int (&rows)[NR], int nvalid,
                        const float *act, int mstride, float *y, const int (&yoff)[NR], int ystride)
{
    const int lane = threadIdx.x & 31;
    const int LPR = lanes_per_row(K), RPP = 32 / LPR;
    float a[SPL][NR][16], as[SPL][NR];
#pragma unroll
    for (int i = 0; i < SPL; ++i) {
        const int sg = lane % LPR + LPR * i;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float4 *src = reinterpret_cast<const float4 *>(act + (size_t)rows[r] * mstride + sg * kSub);
            float s = 0.f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 v = __ldcg(src + t);
                a[i][r][4 * t] = v.x; a[i][r][4 * t + 1] = v.y; a[i][r][4 * t + 2] = v.z; a[i][r][4 * t + 3] = v.w;
                s += (v.x + v.y) + (v.z + v.w);
            }
            as[i][r] = s;
        }
    }
    for (int h0 = 0; h0 < cnt; h0 += RPP * NU) {
        const int hb = h0 + (lane / LPR) * NU;
        const uint8_t *wr[NU];
#pragma unroll
        for (int j = 0; j < NU; ++j) wr[j] = stage + (size_t)(hb + j < cnt ? hb + j : 0) * rowb;
        float acc[NU][NR];
#pragma unroll
        for (int j = 0; j < NU; ++j)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[j][r] = 0.f;
        if (hb < cnt) {
#pragma unroll
            for (int i = 0; i < SPL; ++i)
                rdot_sub<BITS, NR, NU>(wr, K, lane % LPR + LPR * i, a[i], as[i], acc);
        }
        lane_reduce<NU, NR>(acc, LPR);
        if (lane % LPR == 0) {
#pragma unroll
            for (int j = 0; j < NU; ++j)
                if (hb + j < cnt) {
#pragma unroll
                    for (int r = 0; r < NR; ++r)
                        if (r < nvalid) y[yoff[r] + (rs + hb + j) * ystride] = acc[j][r];
                }
        }
    }
}

#define MOE_CASE(BV, RV, CALL) \
    case (BV) * 16 + (RV): { constexpr int B_ = (BV), R_ = (RV); CALL; } break;
#define MOE_CASES_NR(BV, CALL) MOE_CASE(BV, 1, CALL) MOE_CASE(BV, 2, CALL)

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

// Token rows of a mask in groups of up to `gmax`: f(first, NR bucket).
template <typename F>
__device__ __forceinline__ void for_row_groups(uint32_t mask, int gmax, F &&f)
{
    const int n = __popc(mask);
    for (int g0 = 0; g0 < n; g0 += gmax) f(g0, nr_bucket(min(gmax, n - g0)));
}

// One token row: two units (four weight rows) per lane group at a time;
// several token rows: one unit at a time.
__device__ void gu_stage(const Sh &sh, int bits, const uint8_t *stage, int cnt, int rowb, int H, uint32_t mask,
                         float *act, int mstride, int j0)
{
    for_row_groups(mask, 2, [&](int g0, int nr) {
        MOE_DISPATCH(bits, nr, ({
            int rows[R_], nv;
            rows_of_group<R_>(mask, g0, rows, nv);
            // two units at a time for one token row; an odd last unit alone
            const int even = R_ == 1 ? (cnt & ~1) : 0;
            if (even) gu_pass<B_, R_, 2>(sh, stage, even, rowb, H, rows, nv, act, mstride, j0);
            if (cnt > even)
                gu_pass<B_, R_, 1>(sh, stage + (size_t)even * 2 * rowb, cnt - even, rowb, H, rows, nv, act, mstride,
                                   j0 + even);
        }));
    });
}

__device__ void router_stage(const Sh &sh, int bits, const uint8_t *stage, int cnt, int rowb, int H, uint32_t mask,
                             float *logits, int Er, int e0)
{
    for_row_groups(mask, 2, [&](int g0, int nr) {
        MOE_DISPATCH_ROUTER(bits, nr, ({
            int rows[R_], nv;
            rows_of_group<R_>(mask, g0, rows, nv);
            const int even = R_ == 1 ? (cnt & ~1) : 0;
            if (even) router_pass<B_, R_, 2>(sh, stage, even, rowb, H, rows, nv, logits, Er, e0);
            if (cnt > even)
                router_pass<B_, R_, 1>(sh, stage + (size_t)even * rowb, cnt - even, rowb, H, rows, nv, logits, Er,
                                       e0 + even);
        }));
    });
}

// Down rows of one stage for every row group of `mask`.  Routed experts
// write ybuf[(pair0 + r) * hrows + h]; the shared expert writes
// ysh[h * kMaxRows + m].
__device__ void dn_stage(const Sh &sh, int bits, const uint8_t *stage, int rs, int cnt, int rowb, int K, uint32_t mask,
                         const float *act, int mstride, bool shared, int pair0)
{
    const int spl = (K / kSub) / lanes_per_row(K);   // 1 or 2 (K <= 1024)
    const int gmax = 2 / spl;
    for_row_groups(mask, gmax, [&](int g0, int nr) {
        auto run = [&](auto spl_c) {
            constexpr int SPLV = decltype(spl_c)::value;
            MOE_DISPATCH(bits, nr, ({
                if constexpr (R_ * SPLV <= 2) {
                    int rows[R_], nv;
                    rows_of_group<R_>(mask, g0, rows, nv);
                    int yoff[R_];
#pragma unroll
                    for (int r = 0; r < R_; ++r)
                        yoff[r] = shared ? rows[r] : (pair0 + g0 + (r < nv ? r : nv - 1)) * sh.hrows;
                    float *y = shared ? sh.ysh : sh.ybuf;
                    const int ys = shared ? kMaxRows : 1;
                    const int RPPv = 32 / lanes_per_row(K);
                    // pairs of rows per lane group; a leftover row alone
                    const int even = cnt - cnt % (2 * RPPv);
                    if (even) dn_pass<B_, R_, SPLV, 2>(stage, rs, even, rowb, K, rows, nv, act, mstride, y, yoff, ys);
                    if (cnt > even)
                        dn_pass<B_, R_, SPLV, 1>(stage + (size_t)even * rowb, rs + even, cnt - even, rowb, K, rows, nv,
                                                 act, mstride, y, yoff, ys);
                }
            }));
        };
        if (spl == 1) run(std::integral_constant<int, 1>{});
        else run(std::integral_constant<int, 2>{});
    });
}

// ------------------------------------------------------------ P0: RMSNorm

// Per-row sums of squares of M bf16 rows of x (global) into red[], and,
// when `stage` is set, the raw values copied into xs in the arranged layout.
// Then rinv = 1 / sqrt(mean(x^2) + eps) -> red[kMaxRows * kRedChunks + m].
__device__ void rms_rows(const KParams &kp, const Sh &sh, const uint16_t *x, bool stage)
{
    const int H = kp.g.H, M = kp.M, tid = threadIdx.x, lane = tid & 31;
    const int nsg = H / kSub, width = nsg < 32 ? nsg : 32, chunks = nsg / width;
    const int LPR = lanes_per_row(H);
    // pairs are visited in rounds of NCT; all lanes of a warp share a round
    for (int p0 = 0; p0 < M * nsg; p0 += NCT) {
        const int p = p0 + tid;
        float ss = 0.f;
        if (p < M * nsg) {
            const int m = p / nsg, sg = p % nsg;
            const uint4 *xv = reinterpret_cast<const uint4 *>(x + (size_t)m * H + sg * kSub);
            float4 *xs4 = reinterpret_cast<float4 *>(sh.xs + (size_t)m * H);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 a = __ldcg(xv + h);
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f[2 * j] = __uint_as_float(aw[j] << 16);
                    f[2 * j + 1] = __uint_as_float(aw[j] & 0xFFFF0000u);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
                if (stage) {
                    xs4[arr_index(sg, 2 * h, LPR)] = make_float4(f[0], f[1], f[2], f[3]);
                    xs4[arr_index(sg, 2 * h + 1, LPR)] = make_float4(f[4], f[5], f[6], f[7]);
                }
            }
        }
        // sum over the `width` lanes that share a row chunk
        for (int o = width / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULLMASK, ss, o);
        if (p < M * nsg && (lane % width) == 0) {
            const int m = p / nsg, chunk = (p % nsg) / width;
            sh.red[m * kRedChunks + chunk] = ss;
        }
    }
    cbar();
    if (tid < M) {
        float t = 0.f;
        for (int c = 0; c < chunks; ++c) t += sh.red[tid * kRedChunks + c];
        sh.red[kMaxRows * kRedChunks + tid] = rsqrtf(t / (float)H + kp.g.eps);
    }
    cbar();
}

// hn = x * rinv * gamma in the arranged layout, with per-16 sums.
__device__ void build_hn(const KParams &kp, const Sh &sh, const uint16_t *x, const uint16_t *gamma)
{
    const int H = kp.g.H, M = kp.M, tid = threadIdx.x;
    rms_rows(kp, sh, x, true);
    const int nsg = H / kSub, LPR = lanes_per_row(H);
    for (int p = tid; p < M * nsg; p += NCT) {
        const int m = p / nsg, sg = p % nsg;
        const float rinv = sh.red[kMaxRows * kRedChunks + m];
        const uint4 *gv = reinterpret_cast<const uint4 *>(gamma + sg * kSub);
        float4 *xs4 = reinterpret_cast<float4 *>(sh.xs + (size_t)m * H);
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 g = __ldg(gv + h);
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            float4 a = xs4[arr_index(sg, 2 * h, LPR)], b = xs4[arr_index(sg, 2 * h + 1, LPR)];
            a.x = a.x * rinv * __uint_as_float(gw[0] << 16);
            a.y = a.y * rinv * __uint_as_float(gw[0] & 0xFFFF0000u);
            a.z = a.z * rinv * __uint_as_float(gw[1] << 16);
            a.w = a.w * rinv * __uint_as_float(gw[1] & 0xFFFF0000u);
            b.x = b.x * rinv * __uint_as_float(gw[2] << 16);
            b.y = b.y * rinv * __uint_as_float(gw[2] & 0xFFFF0000u);
            b.z = b.z * rinv * __uint_as_float(gw[3] << 16);
            b.w = b.w * rinv * __uint_as_float(gw[3] & 0xFFFF0000u);
            s += ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
            xs4[arr_index(sg, 2 * h, LPR)] = a;
            xs4[arr_index(sg, 2 * h + 1, LPR)] = b;
        }
        sh.xsum[m * nsg + sg] = s;
    }
    for (int e = tid; e < kp.g.E; e += NCT) sh.emask[e] = 0u;
    cbar();
}

// ------------------------------------------------------------- R: routing

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t fkey(float v)
{
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of one row by a warp, keyed on (logit descending, expert id
// ascending).  T = the k-th largest of the 32 lane maxima (a lower bound of
// the k-th largest logit) by an MSB-first radix search with ballots; the
// candidates at or above T (at least k of them) go to shared memory and are
// ranked exactly.  No step depends on a chain of shuffles.
template <int NPL>
__device__ void topk_row_t(const KParams &kp, const Sh &sh, int m, const float *logits)
{
    const int lane = threadIdx.x & 31;
    const int E = kp.g.E, k = kp.g.k, Er = kp.g.Er;
    float v[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcg(logits + (size_t)m * Er + e) : -FLT_MAX;
    }
    const float lsg = kp.g.has_shared ? __ldcg(logits + (size_t)m * Er + E) : 0.f;
    float bv = v[0];
#pragma unroll
    for (int i = 1; i < NPL; ++i) bv = fmaxf(bv, v[i]);
    // k-th largest lane maximum (ties counted with multiplicity)
    const uint32_t key = (lane < E) ? fkey(bv) : 0u;
    uint32_t prefix = 0;
#pragma unroll
    for (int b = 31; b >= 0; --b) {
        const uint32_t trial = prefix | (1u << b);
        if (__popc(__ballot_sync(FULLMASK, key >= trial)) >= k) prefix = trial;
    }
    // candidates: every logit >= T; at least k of them
    unsigned bal[NPL];
    int C = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        bal[i] = __ballot_sync(FULLMASK, lane + 32 * i < E && fkey(v[i]) >= prefix);
        C += __popc(bal[i]);
    }
    float *topv = sh.topv + m * kMaxK;
    int *tope = sh.tope + m * kMaxK;
    if (C <= kCandCap) {
        float *cv = sh.cand_v + m * kCandCap;
        int *ce = sh.cand_e + m * kCandCap;
        int base = 0;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if ((bal[i] >> lane) & 1u) {
                const int pos = base + __popc(bal[i] & ((1u << lane) - 1u));
                cv[pos] = v[i];
                ce[pos] = lane + 32 * i;
            }
            base += __popc(bal[i]);
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
        // many ties at the threshold: k rounds of warp arg-max (exact)
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
            if (lane == 0) { topv[r] = gv; tope[r] = ge < E ? ge : 0; }
        }
    }
    __syncwarp();
    // renormalised softmax weights over the k kept logits (the full softmax
    // probabilities divided by their top-k sum)
    const float vmax = topv[0];
    const float ev = lane < k ? expf(topv[lane] - vmax) : 0.f;
    const float z = warp_sum(ev);
    if (lane < k) {
        const float wv = ev / z;
        sh.topw[m * kMaxK + lane] = wv;
        // the same k entries ordered by expert id (combine order of the row)
        const int e = tope[lane];
        int r = 0;
        for (int j = 0; j < k; ++j) r += tope[j] < e ? 1 : 0;
        sh.row_w[m * kMaxK + r] = wv;
        sh.row_pair[m * kMaxK + r] = e;   // expert id for now; pair index after the slot list
    }
    if (lane == 0) sh.sigma[m] = kp.g.has_shared ? 1.0f / (1.0f + expf(-lsg)) : 0.f;
}

__device__ void topk_row(const KParams &kp, const Sh &sh, int m, const float *logits)
{
    const int E = kp.g.E;
    if (E <= 64) topk_row_t<2>(kp, sh, m, logits);
    else if (E <= 256) topk_row_t<8>(kp, sh, m, logits);
    else topk_row_t<16>(kp, sh, m, logits);
}

__device__ void route(const KParams &kp, const Sh &sh, const float *logits, int l)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = kp.g.E, k = kp.g.k, M = kp.M;
    if (M == 1) {
        // one row: the slots are its k experts in id order
        if (warp == 0) {
            topk_row(kp, sh, 0, logits);
            if (threadIdx.x == 0) stamp(kp, l, 12);
            __syncwarp();
            if (lane < k) {
                const int e = sh.row_pair[lane];
                sh.slot_e[lane] = e;
                sh.slot_mask[lane] = 1u;
                sh.slot_rowbase[lane] = lane;
                sh.row_pair[lane] = lane;
                if (kp.mode == kModeRouter && blockIdx.x == 0) {
                    kp.idx_out[lane] = sh.tope[lane];
                    kp.w_out[lane] = sh.topw[lane];
                }
            }
            if (lane == 0) {
                sh.flags[1] = k;
                sh.slot_rowbase[k] = k;
                stamp(kp, l, 13);
            }
            for (int t = lane; t < k; t += 32) sh.target[t] += (unsigned)kp.g.I;
        }
        cbar();
        return;
    }
    if (warp < M) topk_row(kp, sh, warp, logits);
    if (threadIdx.x == 0) stamp(kp, l, 12);
    cbar();
    if (warp == 0) {
        for (int t = lane; t < M * k; t += 32) {
            const int e = sh.tope[(t / k) * kMaxK + t % k];
            atomicOr(&sh.emask[e < E ? e : 0], 1u << (t / k));
        }
        __syncwarp();
        int base = 0;
        for (int c0 = 0; c0 < E; c0 += 32) {
            const int e = c0 + lane;
            const uint32_t mk = e < E ? sh.emask[e] : 0u;
            const unsigned bal = __ballot_sync(FULLMASK, mk != 0u);
            if (mk) {
                const int pos = base + __popc(bal & ((1u << lane) - 1u));
                sh.slot_e[pos] = e;
                sh.slot_mask[pos] = mk;
                sh.eslot[e] = pos;
            }
            base += __popc(bal);
        }
        __syncwarp();
        // slot-row pair bases: prefix sums of popc(mask) over the slots
        int run = 0;
        for (int s0 = 0; s0 < base; s0 += 32) {
            const int s = s0 + lane;
            const int pc = s < base ? __popc(sh.slot_mask[s]) : 0;
            int inc = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULLMASK, inc, o);
                if (lane >= o) inc += t;
            }
            if (s < base) sh.slot_rowbase[s] = run + inc - pc;
            run += __shfl_sync(FULLMASK, inc, 31);
        }
        if (lane == 0) {
            sh.flags[1] = base;
            sh.slot_rowbase[base] = run;
        }
        for (int t = lane; t < base; t += 32) sh.target[t] += (unsigned)kp.g.I;
        __syncwarp();
        for (int t = lane; t < M * k; t += 32) {
            const int m = t / k, j = t % k;
            const int e = sh.row_pair[m * kMaxK + j];
            const int s = sh.eslot[e < E ? e : 0];
            sh.row_pair[m * kMaxK + j] = sh.slot_rowbase[s] + __popc(sh.slot_mask[s] & ((1u << m) - 1u));
            if (kp.mode == kModeRouter && blockIdx.x == 0) {
                kp.idx_out[m * k + j] = sh.tope[m * kMaxK + j];
                kp.w_out[m * k + j] = sh.topw[m * kMaxK + j];
            }
        }
        if (threadIdx.x == 0) stamp(kp, l, 13);
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

// ------------------------------------------------------------- schedules

// Stage schedule shared by the producer and the compute warps: `f` gets
// (src, bytes, slot-or-kind, first, count) of each stage in order.
template <typename F>
__device__ __forceinline__ void sched_p1(const KParams &kp, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    const int P = gridDim.x, c = blockIdx.x, S = kp.p.S;
    int a, b;
    split(g.Er, P, c, a, b);
    const int cr = S / g.rr_bytes;
    for (int r = a; r < b; r += cr) {
        const int n = min(cr, b - r);
        f(Lp.router + (size_t)r * g.rr_bytes, n * g.rr_bytes, 0, r, n);
    }
    if (kp.mode == kModeLayers && g.has_shared) {
        split(g.Is, P, c, a, b);
        const int ub = 2 * g.sg_bytes;
        const int cu = max(1, min(S / ub, (b - a + NCW - 1) / NCW));
        for (int j = a; j < b; j += cu) {
            const int n = min(cu, b - j);
            f(Lp.sgu + (size_t)j * ub, n * ub, 1, j, n);
        }
    }
}

template <typename F>
__device__ __forceinline__ void sched_p1b(const KParams &kp, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    if (kp.mode != kModeLayers || !g.has_shared) return;
    int h0, h1;
    split(g.H, gridDim.x, blockIdx.x, h0, h1);
    const int nh = h1 - h0;
    const int cd = max(1, min(kp.p.S / g.sd_bytes, (nh + 6) / 7));
    for (int r = 0; r < nh; r += cd) {
        const int n = min(cd, nh - r);
        f(Lp.sdown + (size_t)(h0 + r) * g.sd_bytes, n * g.sd_bytes, -1, r, n);
    }
}

template <typename F>
__device__ __forceinline__ void sched_p2(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    const int U = sh.flags[1];
    const int ub = 2 * g.g_bytes;
    int a, b;
    split(U * g.I, gridDim.x, blockIdx.x, a, b);
    const int cu = max(1, min(kp.p.S / ub, 2 * ((b - a + 2 * NCW - 1) / (2 * NCW))));
    for (int n = a; n < b;) {
        const int s = n / g.I, j = n % g.I;
        const int cnt = min(cu, min(b, (s + 1) * g.I) - n);
        f(Lp.gu + ((size_t)sh.slot_e[s] * g.I + j) * ub, cnt * ub, s, j, cnt);
        n += cnt;
    }
}

template <typename F>
__device__ __forceinline__ void sched_p3(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    const int U = sh.flags[1];
    int h0, h1;
    split(g.H, gridDim.x, blockIdx.x, h0, h1);
    const int nh = h1 - h0;
    const int pieces = max(1, (NCW + U - 1) / max(1, U));
    int cd = max(1, min(kp.p.S / g.d_bytes, (nh + pieces - 1) / pieces));
    if (cd > 1 && (cd & 1)) ++cd;
    cd = min(cd, kp.p.S / g.d_bytes);
    for (int s = 0; s < U; ++s) {
        const int e = sh.slot_e[s];
        for (int r = 0; r < nh; r += cd) {
            const int n = min(cd, nh - r);
            f(Lp.down + ((size_t)e * g.H + h0 + r) * g.d_bytes, n * g.d_bytes, s, r, n);
        }
    }
}

// ------------------------------------------------------------- producer

// Lane `lane` issues the stages q with q % NP == lane.  NS is a multiple of
// NP, so the lane itself issued the previous round of the slot it reuses.
__device__ __forceinline__ bool issue(const Sh &sh, unsigned q, const uint8_t *src, int bytes)
{
    const int slot = (int)(q % (unsigned)sh.NS);
    const unsigned n = q / (unsigned)sh.NS;
    if (n > 0 && !wait_bar(sh, &sh.empty[slot], (n - 1) & 1u, 1)) return false;
    if (aborted(sh)) return false;
    mbar_expect_tx(&sh.full[slot], (unsigned)bytes);
    bulk_load(sh.ring + (size_t)slot * sh.S, src, (unsigned)bytes, &sh.full[slot]);
    return true;
}

__device__ __forceinline__ void producer(const KParams &kp, const Sh &sh, int lane)
{
    unsigned q = 0;
    bool ok = true;
    auto each = [&](const uint8_t *src, int bytes, int, int, int) {
        if (ok && (int)(q % NP) == lane) ok = issue(sh, q, src, bytes);
        ++q;
    };
    for (int l = 0; l < kp.L && ok; ++l) {
        const LayerPtrs &Lp = kp.layer[l];
        sched_p1(kp, Lp, each);
        sched_p1b(kp, Lp, each);
        if (!ok || kp.mode == kModeRouter) break;
        if (lane == 0) stamp(kp, l, 9);
        if (!wait_bar(sh, sh.route, (unsigned)l & 1u, 2)) break;
        if (lane == 0) stamp(kp, l, 10);
        sched_p2(kp, sh, Lp, each);
        sched_p3(kp, sh, Lp, each);
        if (lane == 0) stamp(kp, l, 11);
    }
    // Let this lane's copies still in flight land before the CTA can exit.
    const unsigned first = q > (unsigned)sh.NS ? q - (unsigned)sh.NS : 0u;
    for (unsigned t = first; t < q; ++t) {
        if ((int)(t % NP) != lane) continue;
        const int slot = (int)(t % (unsigned)sh.NS);
        const unsigned long long t0 = now_ns();
        while (!mbar_try_wait(&sh.full[slot], (t / (unsigned)sh.NS) & 1u))
            if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) break;
    }
}

// -------------------------------------------------------- compute warps

// Stage q belongs to warp q % NCW (NS is a multiple of NCW, so the warp
// itself consumed the previous round of the slot before it waits on this one).
template <typename F>
__device__ __forceinline__ void consume(const Sh &sh, unsigned &q, int where, F &&f, const KParams *tk = nullptr,
                                        int tl = 0, int *tcount = nullptr, int tbase = 0, int tmax = 0)
{
    const unsigned me = q++;
    if ((int)(me % NCW) != (int)(threadIdx.x >> 5)) return;
    const int slot = (int)(me % (unsigned)sh.NS);
    const bool st = tk && *tcount < tmax;
    if (st) wstamp(*tk, tl, tbase);
    if (!aborted(sh) && wait_bar(sh, &sh.full[slot], (me / (unsigned)sh.NS) & 1u, where)) {
        if (st) wstamp(*tk, tl, tbase + 1);
        f(sh.ring + (size_t)slot * sh.S);
    }
    __syncwarp();
    if (st) { wstamp(*tk, tl, tbase + 2); ++*tcount; }
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[slot], 1);
}

__device__ void phase1(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w)
{
    const Geo &g = kp.g;
    const uint32_t all = (1u << kp.M) - 1u;
    sched_p1(kp, Lp, [&](const uint8_t *, int, int kind, int first, int n) {
        consume(sh, q, 10, [&](const uint8_t *st) {
            if (kind == 0) router_stage(sh, g.qb, st, n, g.rr_bytes, g.H, all, w.logits, g.Er, first);
            else gu_stage(sh, g.sb, st, n, g.sg_bytes, g.H, all, w.act_s, g.Is, first);
        });
    });
}

__device__ void phase1b(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w, int l)
{
    const Geo &g = kp.g;
    const uint32_t all = (1u << kp.M) - 1u;
    int tc = 0;
    sched_p1b(kp, Lp, [&](const uint8_t *, int, int, int first, int n) {
        consume(sh, q, 15, [&](const uint8_t *st) {
            dn_stage(sh, g.sb, st, first, n, g.sd_bytes, g.Is, all, w.act_s, g.Is, true, 0);
        }, kp.trace ? &kp : nullptr, l, &tc, 11, 1);
    });
}

__device__ void phase2(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w, int l)
{
    const Geo &g = kp.g;
    const int maxr = kp.ws_l.maxr;
    int tc = 0;
    sched_p2(kp, sh, Lp, [&](const uint8_t *, int, int s, int first, int n) {
        consume(sh, q, 20, [&](const uint8_t *st) {
            gu_stage(sh, g.rb, st, n, g.g_bytes, g.H, sh.slot_mask[s], w.act + (size_t)s * maxr * g.I, g.I, first);
            // publish: n more activation units of slot s are in global memory
            // (the warp barrier orders every lane's stores before lane 0's release)
            __syncwarp();
            if ((threadIdx.x & 31) == 0) red_release_add(&sh.act_done[s], (unsigned)n);
        }, kp.trace ? &kp : nullptr, l, &tc, 2, 1);
    });
}

__device__ void phase3(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, unsigned &q, const Ws &w, int l)
{
    const Geo &g = kp.g;
    const int maxr = kp.ws_l.maxr;
    int tc = 0;
    sched_p3(kp, sh, Lp, [&](const uint8_t *, int, int s, int first, int n) {
        consume(sh, q, 30, [&](const uint8_t *st) {
            if (!wait_count(sh, &sh.act_done[s], sh.target[s], 35)) return;
            dn_stage(sh, g.rb, st, first, n, g.d_bytes, g.I, sh.slot_mask[s], w.act + (size_t)s * maxr * g.I, g.I,
                     false, sh.slot_rowbase[s]);
        }, kp.trace ? &kp : nullptr, l, &tc, 7, 1);
    });
}

// out = x + sum_j w_j y_j (expert-id order) + sigma y_shared, for this
// CTA's outputs; thread t holds output (hl, m) = (t / M, t % M).
__device__ void combine(const KParams &kp, const Sh &sh, float xres, uint16_t *xout)
{
    const Geo &g = kp.g;
    const int M = kp.M, k = g.k, t = threadIdx.x;
    int h0, h1;
    split(g.H, gridDim.x, blockIdx.x, h0, h1);
    const int nh = h1 - h0;
    if (t < nh * M) {
        const int hl = t / M, m = t % M;
        float acc = 0.f;
        for (int j = 0; j < k; ++j)
            acc = fmaf(sh.row_w[m * kMaxK + j], sh.ybuf[sh.row_pair[m * kMaxK + j] * sh.hrows + hl], acc);
        if (g.has_shared) acc = fmaf(sh.sigma[m], sh.ysh[hl * kMaxRows + m], acc);
        xout[(size_t)m * g.H + h0 + hl] = f2bf(xres + acc);
    }
}

// out_n = bf16(out * rinv * gamma_next) for this CTA's outputs.
__device__ void write_normed(const KParams &kp, const Sh &sh, const uint16_t *out, const uint16_t *gamma_next)
{
    const Geo &g = kp.g;
    rms_rows(kp, sh, out, false);
    int h0, h1;
    split(g.H, gridDim.x, blockIdx.x, h0, h1);
    const int nh = h1 - h0, M = kp.M;
    for (int t = threadIdx.x; t < nh * M; t += NCT) {
        const int hl = t / M, m = t % M;
        const size_t idx = (size_t)m * g.H + h0 + hl;
        const float v = bf2f(__ldcg(out + idx)) * sh.red[kMaxRows * kRedChunks + m] * bf2f(gamma_next[h0 + hl]);
        kp.out_normed[idx] = f2bf(v);
    }
}

__device__ __forceinline__ void compute(const KParams &kp, const Sh &sh)
{
    const Ws w = ws_views(kp);
    unsigned q = 0;
    int nsync = 0;
    int h0, h1;
    split(kp.g.H, gridDim.x, blockIdx.x, h0, h1);
    const int nh = h1 - h0;
    for (int l = 0; l < kp.L; ++l) {
        const LayerPtrs &Lp = kp.layer[l];
        const bool last = l == kp.L - 1;
        const uint16_t *xin = l == 0 ? kp.x : w.ping[(l - 1) & 1];
        uint16_t *xout = last ? kp.out : w.ping[l & 1];
        const bool t0 = threadIdx.x == 0;
        if (t0) stamp(kp, l, 0);
        build_hn(kp, sh, xin, Lp.gamma);
        if (t0) stamp(kp, l, 1);
        phase1(kp, sh, Lp, q, w);
        if (t0) stamp(kp, l, 2);
        if (!grid_sync(kp, sh, nsync)) return;
        if (t0) stamp(kp, l, 3);
        route(kp, sh, w.logits, l);
        if (t0) stamp(kp, l, 4);
        if (kp.mode == kModeRouter) break;
        if (t0) mbar_arrive(sh.route, 1);
        // residual of this thread's output, read while the weights stream
        float xres = 0.f;
        if ((int)threadIdx.x < nh * kp.M) {
            const int hl = threadIdx.x / kp.M, m = threadIdx.x % kp.M;
            xres = bf2f(__ldcg(xin + (size_t)m * kp.g.H + h0 + hl));
        }
        wstamp(kp, l, 0);
        phase1b(kp, sh, Lp, q, w, l);
        wstamp(kp, l, 1);
        phase2(kp, sh, Lp, q, w, l);
        wstamp(kp, l, 5);
        if (t0) stamp(kp, l, 5);
        if (t0) stamp(kp, l, 6);
        wstamp(kp, l, 6);
        phase3(kp, sh, Lp, q, w, l);
        wstamp(kp, l, 10);
        if (cbar_or(aborted(sh))) return;
        combine(kp, sh, xres, xout);
        if (t0) stamp(kp, l, 7);
        if (!last || kp.out_normed) {
            if (!grid_sync(kp, sh, nsync)) return;
        }
        if (t0) stamp(kp, l, 8);
        if (last && kp.out_normed) write_normed(kp, sh, xout, Lp.gamma_next);
    }
    kernel_exit(sh, kp.p.max_slots);
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
    sh.sigma = reinterpret_cast<float *>(smem + L.sigma);
    sh.eslot = reinterpret_cast<int *>(smem + L.eslot);
    sh.emask = reinterpret_cast<uint32_t *>(smem + L.emask);
    sh.topv = reinterpret_cast<float *>(smem + L.topv);
    sh.tope = reinterpret_cast<int *>(smem + L.tope);
    sh.topw = reinterpret_cast<float *>(smem + L.topw);
    sh.row_w = reinterpret_cast<float *>(smem + L.row_w);
    sh.row_pair = reinterpret_cast<int *>(smem + L.row_pair);
    sh.cand_v = reinterpret_cast<float *>(smem + L.cand_v);
    sh.cand_e = reinterpret_cast<int *>(smem + L.cand_e);
    sh.red = reinterpret_cast<float *>(smem + L.red);
    sh.xs = reinterpret_cast<float *>(smem + L.xs);
    sh.xsum = reinterpret_cast<float *>(smem + L.xsum);
    sh.ybuf = reinterpret_cast<float *>(smem + L.ybuf);
    sh.ysh = reinterpret_cast<float *>(smem + L.ysh);
    sh.target = reinterpret_cast<unsigned *>(smem + L.target);
    sh.act_done = reinterpret_cast<unsigned *>(kp.ws + kFlagsOffset);
    sh.ring = smem + L.ring;
    sh.NS = kp.p.NS;
    sh.S = kp.p.S;
    sh.hrows = kp.p.hrows;
    sh.timeout_ns = kp.timeout_ns;
    sh.ctrl = reinterpret_cast<Ctrl *>(kp.ws);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kp.p.NS; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(sh.route, 1);
        sh.flags[0] = 0;
        sh.flags[1] = 0;
        for (int i = 0; i < kp.p.max_slots; ++i) sh.target[i] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= NCT) {
        const int lane = threadIdx.x - NCT;
        if (lane < NP) producer(kp, sh, lane);
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
    p.hrows = (g.H + num_sms - 1) / num_sms;
    int maxi = g.rr_bytes;
    if (2 * g.g_bytes > maxi) maxi = 2 * g.g_bytes;
    if (g.d_bytes > maxi) maxi = g.d_bytes;
    if (g.has_shared) {
        if (2 * g.sg_bytes > maxi) maxi = 2 * g.sg_bytes;
        if (g.sd_bytes > maxi) maxi = g.sd_bytes;
    }
    // Every stage has one consumer warp: stage q goes to warp q % NCW, and a
    // warp waits on stage q only after it waited on stage q - NS of the same
    // slot (mbarrier parity tells apart only the current and previous phase),
    // so NS is a multiple of NCW (and of NP, for the issuing lanes).
    static_assert(NCW % NP == 0, "producer lanes must divide the ring depth");
    for (int ns = 2 * NCW; ns >= NCW; ns -= NCW) {
        p.NS = ns;
        p.S = 16;
        const int fixed = carve(g, p).ring;
        int S = (kSmemMax - fixed - 256) / ns;
        S -= S % 16;
        if (S < maxi) continue;
        p.S = S;
        p.smem_bytes = carve(g, p).total;
        if (p.smem_bytes <= kSmemMax) return true;
    }
    return false;
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
