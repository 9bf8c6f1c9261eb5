// Persistent decode kernel of the quantized MoE FFN layer (and of a stack of
// such layers) for sm_103a.
//
// One CTA per SM: eleven compute warps (launches of at most 4 rows of at
// most 2048 inputs) or eight (this source compiled with MOE_NCW=8), and one
// producer warp.  The producer
// streams weights into shared memory with 1-D bulk copies
// (cp.async.bulk ... mbarrier::complete_tx): a ring of stages holding the
// routed experts (and shared-expert rows that do not fit elsewhere), each
// stage consumed by one compute warp, issued one lane per stage so that the
// copies of a layer go out together; and a prefetch buffer with the next
// layer's RMSNorm weight, the CTA's column slice of the router and
// shared-expert rows, which do not depend on routing and are therefore loaded while the current layer still
// runs.  Per layer:
//
//   P0  every CTA: partial router dots -- every router row dotted with
//       gamma * x over the CTA's own output slice of the layer input (its
//       own output of the previous layer), and x^2 summed over the slice --
//       published as tagged words (flash-moe, "Metal Compute Shaders": RMS
//       normalisation; PureDrive model card, "Summary": 256 experts plus
//       the shared expert's gate)
//   P1  the first M warps, one token row each: the CTA's router rows summed
//       over every CTA's partials and published, then softmax + top-k +
//       renormalisation on every CTA's logits scaled by the row's
//       1 / rms, and the list of distinct selected experts with the rows
//       that chose each (model card, "Summary": the full top-8 of 256 is
//       kept); meanwhile the other warps gather the whole input, build its
//       RMSNorm into shared memory and compute this CTA's shared-expert
//       gate/up units and their SwiGLU
//   P2  gate/up units of the selected experts, each expert streamed once for
//       all the rows that chose it (model card, "How it works": the verify
//       pass reads its weights once), SwiGLU
//   S   the shared expert's down rows of this CTA's output slice
//   P3  down rows of every selected expert for this CTA's output slice
//   C   weighted combine + sigmoid-gated shared expert + residual, bf16
//       (flash-moe: "MoE combine + residual + gate")
//   N   the fused next RMSNorm of the bf16 output (model card: fused
//       add+RMSNorm), or the next layer's P0.
//
// CTAs exchange data (partial router dots, router logits, activations,
// layer outputs) as tagged words in global memory that readers poll, a
// whole warp's missing words per round; there is no grid barrier between
// phases or layers.
//
// Dequantisation (moe_unpack.cuh).  A lane takes one 64-code group of a
// weight row.  A masked code read as a float is the subnormal
// q * 2^(p - 149); the activations sit in shared memory multiplied by
// 2^100, so a paired FFMA2 of masked codes against them accumulates
// q * x * 2^(p - 49) as exact fp32 products.  Codes are accumulated per bit
// position ("class") and each class sum is scaled back once per group: one
// LOP3 and half an FFMA2 per weight and token row.  The affine terms are
// factored per group: sum_j (q_j s + b) x_j = s * sum_j q_j x_j + b * sum_j x_j.
//
// Determinism: no float atomics; every sum has a fixed order that depends
// only on the row itself, so row m of an M-row call equals a 1-row call.
#include <cuda_bf16.h>

#include <cfloat>
#include <climits>
#include <cstring>
#include <mutex>

#include "moe_internal.h"
#include "moe_unpack.cuh"

namespace moe {
namespace {

// Compute warps of this build (the library builds 11 and 8: decode_plan).
#ifndef MOE_NCW
#define MOE_NCW 11
#endif
#if MOE_NCW == 11
#define MOE_WBUILD(name) name
#else
#define MOE_WBUILD(name) name##_w8
#endif
constexpr int NCW = MOE_NCW;
constexpr int NCT = NCW * 32;
constexpr int kThreads = (NCW + 1) * 32;   // + the producer warp
constexpr unsigned FULLMASK = 0xffffffffu;
constexpr float kXScale = 0x1p100f;  // arranged vectors hold x * 2^100
// RMSNorm sums of squares: one slot per 256 inputs of a row (H <= 8192),
// then 1 / rms
constexpr int kSsChunks = 32;
constexpr int kRed = kSsChunks + 1;

// ------------------------------------------------------------ shared layout

// Per-CTA constants of a launch, computed once into shared memory: this
// CTA's router rows, shared gate/up units and output slice, and what its
// prefetch buffer holds.  The prefetch buffer of a layer is gamma, the
// CTA's slice of the input-major router (the columns of its output slice,
// every row), the shared expert's down rows of the output slice (when they
// fit) and as many of the shared units as fit; the rest go through the ring.
struct CtaPlan {
    int ra, rb;        // router rows (row Er: the sum of squares) this CTA sums and publishes
    int ua, ub;        // shared units of this CTA
    int upb;           // units held in the buffer: [ua, ua + upb)
    int h0, nh;        // output slice (whole row pairs): rows h0 .. h0 + nh
    int dpb;           // shared down rows held in the buffer: nh or 0
    int g0, ng;        // groups the slice touches: g0 .. g0 + ng
    int off_router;    // router codes (or fp32 values) of the slice: [nh][Erp]
    int off_rsb;       // their scale/bias words: [ng][Erp]
    int off_sdown, off_units, bytes;
};

// Bytes reserved for the CTA's Sh (pointers into shared memory and launch
// constants), which lives in shared memory itself.
constexpr int kShBytes = 512;

struct SmemLayout {
    int shs, cplan, bar, flags, slot_e, slot_mask, slot_rowbase, sigma, eslot, emask, topv, tope, topw;
    int row_w, row_pair, red, ru, pair_src, xs, xsum, act, asum, ysh, yl, pb, ring, total;
};

__host__ __device__ inline int take(int &o, int bytes, int align)
{
    o = (int)align_up((size_t)o, (size_t)align);
    const int r = o;
    o += bytes;
    return r;
}

__host__ __device__ inline int imax_of(const Geo &g) { return g.Is > g.I ? g.Is : g.I; }

// Router rows (logits summed) / shared units taken by one CTA at most.
__host__ __device__ inline int per_cta(int n, int P) { return (n + P - 1) / P; }

__host__ __device__ inline SmemLayout carve(const Geo &g, const Plan &p)
{
    SmemLayout L;
    int o = 0;
    const int ms = p.max_slots, Im = imax_of(g);
    L.shs = take(o, kShBytes, 16);
    L.cplan = take(o, (int)sizeof(CtaPlan), 16);
    L.bar = take(o, (2 * p.NS + 3) * 8, 8);
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
    L.red = take(o, kMaxRows * kRed * 4, 4);
    L.ru = take(o, 2 * kMaxRows * p.hrows * 4, 16);
    L.pair_src = take(o, p.act_pairs * 4, 4);
    L.xs = take(o, p.maxr * g.H * 4, 16);
    L.xsum = take(o, p.maxr * (g.H / kGroup) * 4, 16);
    L.act = take(o, p.act_pairs * Im * 4, 16);
    L.asum = take(o, p.act_pairs * (Im / kGroup) * 4, 16);
    L.ysh = take(o, p.hrows * kMaxRows * 4, 16);
    L.yl = take(o, p.maxr * g.k * p.hrows * 4, 16);
    L.pb = take(o, p.pb_bytes, 128);
    L.ring = take(o, p.NS * p.S, 128);
    L.total = o;
    return L;
}

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

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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

// L2 policy for the weight stream: every weight byte is read once per pass,
// so its lines go first when L2 needs room; the kernel's code, activations,
// logits and counters then stay resident instead of being pushed out to
// HBM by the 26 GB of weights that pass through L2 on every stack forward.
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(evict_first_policy())
                 : "memory");
}

// Starts moving `bytes` (a multiple of 16; src 16-byte aligned) from global
// memory into L2, with no completion signal.
__device__ __forceinline__ void prefetch_l2(const void *src, unsigned bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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

__device__ __forceinline__ void st_relaxed(unsigned *p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Tagged words: a 32-bit payload (an fp32 value, or two bf16 values) with
// the 32-bit tag of the layer that wrote it, stored and loaded as one
// 64-bit access.  A reader that sees its own layer's tag has the value; no
// separate flag, counter or barrier is needed to publish data between CTAs.

__device__ __forceinline__ void st_tag(uint64_t *p, uint32_t payload, unsigned tag)
{
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(((uint64_t)tag << 32) | payload) : "memory");
}

__device__ __forceinline__ uint64_t ld_tag(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Two adjacent tagged words (p 16-byte aligned) in one access.
__device__ __forceinline__ void ld_tag2(const uint64_t *p, uint64_t &a, uint64_t &b)
{
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf(float v)
{
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&h);
}

// A code below 2^23 as a float without an int-to-float conversion: placed
// in the mantissa of 2^23 and 2^23 subtracted (the magic-number conversion
// of quantised GEMM kernels, e.g. Kim et al. 2022).  Exact.
__device__ __forceinline__ float code_float(uint32_t q) { return __uint_as_float(q | 0x4B000000u) - 8388608.0f; }

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
// stored after the per-CTA stamps: [2][kMaxLayers][16 warp slots][16 events].
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
    const CtaPlan *cp;
    uint64_t *full, *empty, *route, *pb_full, *pb_empty;
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
    float *red;          // [kMaxRows][kRed] RMSNorm sums of 256-input chunks, then 1/rms
    float *ru;           // [2][kMaxRows][hrows] the CTA's input slice: gamma * x, then x
    int *pair_src;       // [act_pairs] slot * kMaxRows + row of each staged pair
    float4 *xs;          // [maxr][H / 4] arranged hn * 2^100
    float *xsum;         // [maxr][H / 64] group sums of hn
    float4 *act;         // [act_pairs][K / 4] arranged activations * 2^100
    float *asum;         // [act_pairs][K / 64]
    float *ysh;          // [hrows][kMaxRows] shared expert outputs
    float *yl;           // [pairs][hrows] routed expert outputs of this CTA's output rows
    uint8_t *pb;
    uint8_t *ring;
    int NS, S, hrows, act_pairs;
    long long timeout_ns;
    Ctrl *ctrl;
    unsigned epoch;      // tags of this launch: epoch + layer + 1 (epoch = launch sequence * 64)
};
static_assert(sizeof(Sh) <= kShBytes, "Sh does not fit its shared-memory slot");

// Tag of the words layer l of this launch publishes.  The launch sequence
// number lives in the workspace control block and advances when a launch
// ends, so every launch has tags of its own even when its parameters are
// the same as an earlier launch's (a replayed launch, a CUDA graph).
__device__ __forceinline__ unsigned layer_tag(const Sh &sh, int l) { return sh.epoch + (unsigned)l + 1u; }


__device__ __forceinline__ bool aborted(const Sh &sh) { return *(volatile int *)&sh.flags[0] != 0; }

// Bounds-checked build (compiled with MOE_DEBUG_BOUNDS): an index computed
// from data (an expert id out of the top-k, a slot or pair number) is
// compared with the size of what it indexes before it is used; one out of
// range sets kStatusBounds in the status word, records 1000 + site in
// `where`, and is replaced by 0 so that the access stays inside its array
// and the launch runs to its end (the host then returns MOE_ERR_DEVICE).
// In the normal build the check is the identity.
#ifdef MOE_DEBUG_BOUNDS
__device__ __noinline__ void bounds_fail(const Sh &sh, int site)
{
    atomicOr(&sh.ctrl->status, kStatusBounds);
    atomicExch(&sh.ctrl->where, 1000 + site);
}
__device__ __forceinline__ int chk(const Sh &sh, int v, int lim, int site)
{
    if ((unsigned)v < (unsigned)lim) return v;
    bounds_fail(sh, site);
    return 0;
}
#else
__device__ __forceinline__ int chk(const Sh &, int v, int, int) { return v; }
#endif

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

// Bookkeeping of a bounded poll: false once the wait ran out (the abort flag
// is then raised) or another thread gave up.  `it` counts failed rounds.
__device__ __forceinline__ bool poll_more(const Sh &sh, unsigned it, unsigned long long &t0, int where)
{
    if (it == 1) t0 = now_ns();
    else if ((it & 15) == 0) {
        if (aborted(sh)) return false;
        if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) {
            raise_abort(sh, where);
            return false;
        }
    }
    __nanosleep(32);
    return true;
}

// N items of four consecutive tagged words each (16-byte aligned; null for
// no item): payloads into out[n].  All words are loaded together, then in
// each round the warp loads again every pair of words that is still
// missing, until no lane misses any: the rounds are the whole warp's, one
// memory round trip each, so that no lane's wait is serialised behind
// another's.  Every lane of the warp takes part.  Bounded (poll_more);
// payloads are 0 after a timeout.
template <int N>
__device__ __forceinline__ void poll_items(const Sh &sh, const uint64_t *const (&p)[N], unsigned tag, int where,
                                           uint32_t (&out)[N][4])
{
    const uint64_t none = (uint64_t)tag << 32;
    uint64_t v[N][4];
#pragma unroll
    for (int n = 0; n < N; ++n) {
        v[n][0] = v[n][1] = v[n][2] = v[n][3] = none;
        if (p[n]) { ld_tag2(p[n], v[n][0], v[n][1]); ld_tag2(p[n] + 2, v[n][2], v[n][3]); }
    }
    unsigned long long t0 = 0;
    unsigned it = 0;
#pragma unroll 1
    for (;;) {
        bool missing = false;
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) missing |= (unsigned)(v[n][j] >> 32) != tag;
        if (!__any_sync(FULLMASK, missing)) break;
        if (!__all_sync(FULLMASK, poll_more(sh, ++it, t0, where))) {
#pragma unroll
            for (int n = 0; n < N; ++n) v[n][0] = v[n][1] = v[n][2] = v[n][3] = 0;
            break;
        }
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int j = 0; j < 4; j += 2)
                if ((unsigned)(v[n][j] >> 32) != tag || (unsigned)(v[n][j + 1] >> 32) != tag)
                    ld_tag2(p[n] + j, v[n][j], v[n][j + 1]);
    }
#pragma unroll
    for (int n = 0; n < N; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) out[n][j] = (uint32_t)v[n][j];
}

// End of a launch for one CTA (thread 0, once its compute warps are done,
// whether or not a wait gave up): the last CTA to finish advances the
// workspace's launch sequence, so that the next launch's tags differ from
// every tag of this one.  When the sequence wraps, that CTA first clears
// every tagged word of the workspace (no CTA of this launch reads them any
// more), so that no word an earlier launch wrote can carry a later tag.
__device__ void kernel_exit(const KParams &kp, const Sh &sh)
{
    Ctrl *ctrl = sh.ctrl;
    const unsigned old = atom_add_acqrel(&ctrl->exit, 1u);
    if (old != gridDim.x - 1) return;
    st_relaxed(&ctrl->exit, 0u);
    unsigned next = sh.epoch / 64u + 1u;
    if (next >= kSeqWrap) {
        uint4 *p = reinterpret_cast<uint4 *>(kp.ws + kp.ws_l.off_logits);
        uint4 *const end = reinterpret_cast<uint4 *>(kp.ws + kp.ws_l.off_stage_in);
#pragma unroll 1
        for (; p < end; ++p) *p = make_uint4(0u, 0u, 0u, 0u);
        __threadfence();
        next = 0u;
    }
    st_relaxed(&ctrl->seq, next);
}

// Part c of P of n items: [n c / P, n (c + 1) / P).  n P < 2^32 (the host
// plan checks the largest n).
__device__ __forceinline__ void split(int n, int P, int c, int &a, int &b)
{
    a = (int)((unsigned)n * (unsigned)c / (unsigned)P);
    b = (int)((unsigned)n * (unsigned)(c + 1) / (unsigned)P);
}

// This CTA's output rows [h0, h1): whole pairs of rows, so that a row pair of
// bf16 outputs goes out as one tagged word.
__device__ __forceinline__ void hslice(int H, int &h0, int &h1)
{
    split(H / 2, gridDim.x, blockIdx.x, h0, h1);
    h0 *= 2;
    h1 *= 2;
}

// ------------------------------------------------------ dequant + dot kernels

__device__ __forceinline__ int ilog2(int x) { return 31 - __clz(x); }

// Arranged vectors: for K inputs in G = K / 64 groups, float4 number
// t * G + g holds inputs 64 g + 4 t .. 64 g + 4 t + 3 (times 2^100), so the
// lanes of a warp, one group each, read consecutive float4s.

// Codes of group g of a packed row (64 codes, 8 * BITS bytes).
// Shared-memory loads by 32-bit shared address: the row kernels are not
// inlined into the kernel, so generic pointers would not be known to point
// to shared memory.
__device__ __forceinline__ uint4 lds4(uint32_t a)
{
    uint4 v;
    asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 ldsf4(uint32_t a)
{
    float4 v;
    asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds1(uint32_t a)
{
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float ldsf1(uint32_t a)
{
    float v;
    asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

template <int BITS>
__device__ __forceinline__ void load_group(uint32_t row, int g, uint32_t (&w)[2 * BITS])
{
#pragma unroll
    for (int i = 0; i < BITS / 2; ++i) {
        const uint4 v = lds4(row + g * 8 * BITS + 16 * i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
}

__device__ __forceinline__ void scale_bias(uint32_t row, int K, int bits, int g, float &s, float &b)
{
    const uint32_t sbw = lds1(row + K * bits / 8 + g * 4);
    s = __uint_as_float(sbw << 16);
    b = __uint_as_float(sbw & 0xFFFF0000u);
}

__device__ __forceinline__ float2 xpair(const float4 &x, int half)
{
    return half ? make_float2(x.z, x.w) : make_float2(x.x, x.y);
}

// First pair of class c (pairs of one class share both positions).
template <typename PT>
__host__ __device__ constexpr int first_of_class(int c)
{
    int i0 = 0;
    for (int i = 7; i >= 0; --i)
        if (PT::cls(i) == c) i0 = i;
    return i0;
}

// Chunk order of a lane.  At 8 and 4 bits a group is 64 or 32 bytes, so
// the same 16-byte chunk of neighbouring lanes' groups falls on the same
// shared-memory banks; each lane starts at a different chunk instead.  (At
// 6 bits the 48-byte stride already spreads the banks.)
template <int BITS>
__device__ __forceinline__ int chunk_rot(int g)
{
    return BITS == 8 ? (g >> 1) & 3 : BITS == 4 ? (g >> 2) & 1 : 0;
}

__device__ __forceinline__ uint2 lds2(uint32_t a)
{
    uint2 v;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// Visits the 4 sub-groups of group g of NROWS rows: f(sg, parity, words[n])
// with words[n] the sub-group's BITS/2 code words of row n and parity a
// compile-time visit parity (0, 1).  Two sub-groups per loop trip, the loop
// not unrolled: the kernel's code then stays small enough to remain in the
// instruction caches between layers.
template <int BITS, int NROWS, typename F>
__device__ __forceinline__ void for_subgroups(const uint32_t (&rp)[NROWS], int g, F &&f)
{
    if constexpr (BITS == 6) {
        // 24 bytes (two sub-groups) per trip; lanes 8 .. 15 of each half warp
        // start with the other pair so that 8-byte loads spread the banks
        const int rot = (g >> 3) & 1;
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            const int jj = j ^ rot;
            uint32_t w[NROWS][6];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) {
                const uint32_t a = rp[n] + g * 48 + 24 * jj;
                const uint2 v0 = lds2(a), v1 = lds2(a + 8), v2 = lds2(a + 16);
                w[n][0] = v0.x; w[n][1] = v0.y; w[n][2] = v1.x; w[n][3] = v1.y; w[n][4] = v2.x; w[n][5] = v2.y;
            }
            const uint32_t *w0[NROWS], *w1[NROWS];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) { w0[n] = &w[n][0]; w1[n] = &w[n][3]; }
            f(2 * jj, 0, w0);
            f(2 * jj + 1, 1, w1);
        }
    } else if constexpr (BITS == 8) {
        // one 16-byte chunk per sub-group, two per trip
        const int rot = chunk_rot<8>(g);
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            const int c0 = (2 * j + rot) & 3, c1 = (2 * j + 1 + rot) & 3;
            uint32_t w[NROWS][8];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) {
                const uint4 v0 = lds4(rp[n] + g * 64 + 16 * c0), v1 = lds4(rp[n] + g * 64 + 16 * c1);
                w[n][0] = v0.x; w[n][1] = v0.y; w[n][2] = v0.z; w[n][3] = v0.w;
                w[n][4] = v1.x; w[n][5] = v1.y; w[n][6] = v1.z; w[n][7] = v1.w;
            }
            const uint32_t *w0[NROWS], *w1[NROWS];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) { w0[n] = &w[n][0]; w1[n] = &w[n][4]; }
            f(c0, 0, w0);
            f(c1, 1, w1);
        }
    } else {
        // 4 bits: a 16-byte chunk holds two sub-groups
        const int rot = chunk_rot<4>(g);
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            const int c = (j + rot) & 1;
            uint32_t w[NROWS][4];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) {
                const uint4 v = lds4(rp[n] + g * 32 + 16 * c);
                w[n][0] = v.x; w[n][1] = v.y; w[n][2] = v.z; w[n][3] = v.w;
            }
            const uint32_t *w0[NROWS], *w1[NROWS];
#pragma unroll
            for (int n = 0; n < NROWS; ++n) { w0[n] = &w[n][0]; w1[n] = &w[n][2]; }
            f(2 * c, 0, w0);
            f(2 * c + 1, 1, w1);
        }
    }
}

// acc[n][r] += dot(row n, group g) . x_r for NROWS weight rows and NR token
// rows, with per-class accumulators (split by visit parity at 4 and 8 bits,
// which have few classes, for more independent chains).  The codes are
// extracted once for all token rows; each token row's arithmetic is the
// same whatever NR is, so a row's result does not depend on the other rows
// of the call (row-exact).
template <int BITS, int NROWS, int NR>
__device__ __forceinline__ void grp_cls(const uint32_t (&rp)[NROWS], int g, int K, int G, const uint32_t (&xq)[NR],
                                        const float (&xsum)[NR], float (&acc)[NROWS][NR])
{
    using PT = Pairs<BITS>;
    constexpr int NC = PT::NC, NA = BITS == 6 ? NC : 2 * NC;
    float s[NROWS], b[NROWS];
#pragma unroll
    for (int n = 0; n < NROWS; ++n) scale_bias(rp[n], K, BITS, g, s[n], b[n]);
    float2 A[NROWS][NR][NA];
#pragma unroll
    for (int n = 0; n < NROWS; ++n)
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int c = 0; c < NA; ++c) A[n][r][c] = make_float2(0.f, 0.f);
    const uint32_t G16 = G * 16;
    for_subgroups<BITS, NROWS>(rp, g, [&](int sg, int step, const uint32_t *const (&ws)[NROWS]) {
        float4 xv[NR][4];
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int t = 0; t < 4; ++t) xv[r][t] = ldsf4(xq[r] + g * 16 + (4 * sg + t) * G16);
        const int half = NA > NC ? step * NC : 0;
#pragma unroll
        for (int n = 0; n < NROWS; ++n)
            PT::each(ws[n], [&](int i, float a, float bb) {
                const float2 q = make_float2(a, bb);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    A[n][r][PT::cls(i) + half] =
                        __ffma2_rn(q, xpair(xv[r][i >> 1], i & 1), A[n][r][PT::cls(i) + half]);
            });
    });
#pragma unroll
    for (int n = 0; n < NROWS; ++n)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float t = 0.f;
#pragma unroll
            for (int c = 0; c < NA; ++c) {
                const int i0 = first_of_class<PT>(c % NC);
                t = fmaf(A[n][r][c].x, __uint_as_float(cls_bits(PT::pa(i0))), t);
                t = fmaf(A[n][r][c].y, __uint_as_float(cls_bits(PT::pb(i0))), t);
            }
            acc[n][r] = fmaf(s[n], t, fmaf(b[n], xsum[r], acc[n][r]));
        }
}

// fp32 rows (a router given in fp32): K floats per row.
template <int NROWS, int NR>
__device__ __forceinline__ void grp_f32(const uint32_t (&rp)[NROWS], int g, int G,
                                        const uint32_t (&xq)[NR], float (&acc)[NROWS][NR])
{
#pragma unroll
    for (int n = 0; n < NROWS; ++n) {
        float S[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) S[r] = 0.f;
#pragma unroll 4
        for (int t = 0; t < 16; ++t) {
            const float4 wq = ldsf4(rp[n] + (g * 16 + t) * 16);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float4 x = ldsf4(xq[r] + (t * G + g) * 16);
                S[r] = fmaf(wq.x, x.x, fmaf(wq.y, x.y, fmaf(wq.z, x.z, fmaf(wq.w, x.w, S[r]))));
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[n][r] = fmaf(S[r], 0x1p-100f, acc[n][r]);
    }
}

// A warp computes rows [0, nrows) (row i at base + i * rstride, K inputs
// at BITS bits) against NR arranged token vectors.  Lanes split a row's
// groups (LPR lanes per row, GPL groups per lane); each lane takes NROWS
// consecutive rows.  emit(first_row, acc) runs on the first lane of each
// row group with the complete sums of rows first_row .. first_row+NROWS-1
// (rows at or past nrows hold repeats of the last row and must be ignored).
template <int BITS, int NROWS, int NR, typename F>
__device__ __forceinline__ void warp_rows(const uint8_t *base, int rstride, int nrows, int K,
                                          const uint32_t (&xq)[NR], const float (&xsg)[NR][kMaxGPL],
                                          F &&emit)
{
    const int lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(base);
    // K and G are powers of two: shifts instead of divisions
    const int G = K >> 6, lgG = ilog2(G), lgL = lgG < 5 ? lgG : 5;
    const int LPR = 1 << lgL, GPL = G >> lgL, RPP = 32 >> lgL;
    const int lg = lane & (LPR - 1), lr = lane >> lgL;
    for (int r0 = 0; r0 < nrows; r0 += RPP * NROWS) {
        const int rb = r0 + lr * NROWS;
        uint32_t rp[NROWS];
#pragma unroll
        for (int n = 0; n < NROWS; ++n) rp[n] = sbase + (uint32_t)(min(rb + n, nrows - 1) * rstride);
        float acc[NROWS][NR];
#pragma unroll
        for (int n = 0; n < NROWS; ++n)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[n][r] = 0.f;
        if (rb < nrows) {
            for (int j = 0; j < GPL; ++j) {
                const int g = lg + LPR * j;
                if constexpr (BITS == 0) {
                    grp_f32<NROWS, NR>(rp, g, G, xq, acc);
                } else {
                    float xs[NR];
#pragma unroll
                    for (int r = 0; r < NR; ++r) xs[r] = xsg[r][j];
                    grp_cls<BITS, NROWS, NR>(rp, g, K, G, xq, xs, acc);
                }
            }
        }
        for (int o = LPR >> 1; o >= 1; o >>= 1)
#pragma unroll
            for (int n = 0; n < NROWS; ++n)
#pragma unroll
                for (int r = 0; r < NR; ++r) acc[n][r] += __shfl_xor_sync(FULLMASK, acc[n][r], o);
        if (lg == 0 && rb < nrows) emit(rb, acc);
    }
}

// Per-lane group sums of NR arranged vectors (sums[soff[r] + g] layout).
template <int NR>
__device__ __forceinline__ void lane_gsums(uint32_t sums, const int (&soff)[NR], int K, float (&xsg)[NR][kMaxGPL])
{
    const int lane = threadIdx.x & 31;
    const int G = K >> 6, lgG = ilog2(G), lgL = lgG < 5 ? lgG : 5;
    const int LPR = 1 << lgL, GPL = G >> lgL, lg = lane & (LPR - 1);
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int j = 0; j < kMaxGPL; ++j) xsg[r][j] = j < GPL ? ldsf1(sums + 4 * (soff[r] + lg + LPR * j)) : 0.f;
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

// Row groups of a mask: pairs, then a single row.
template <typename F>
__device__ __forceinline__ void for_row_groups(uint32_t mask, F &&f)
{
    const int n = __popc(mask);
    int g0 = 0;
    for (; n - g0 >= 2; g0 += 2) f(g0, 2);
    if (n - g0 == 1) f(g0, 1);
}

// The warp-level row kernels below are separate (not inlined) functions,
// one per (bits, token rows): each gets its own register allocation, and a
// call is made once per stage and row group, not per weight.

// Gate/up units [0, cnt) at `units` (unit u: gate row then up row, row
// bytes rowb, K = H inputs) for token rows g0 .. of `mask` against hn:
// dst[m * ld + u] = silu(gate) * up.
template <int B, int R>
__device__ __forceinline__ void gu_k_body(const float4 *xs, const float *xsum, int H, const uint8_t *units, int cnt,
                                  int rowb, uint32_t mask, int g0, uint64_t *dst, int ld, size_t cs, unsigned tag)
{
    const int G = H / kGroup;
    int rows[R], nv;
    rows_of_group<R>(mask, g0, rows, nv);
    uint32_t xq[R];
    int soff[R];
#pragma unroll
    for (int r = 0; r < R; ++r) { xq[r] = smem_u32(xs) + (uint32_t)(rows[r] * H * 4); soff[r] = rows[r] * G; }
    float xsg[R][kMaxGPL];
    lane_gsums<R>(smem_u32(xsum), soff, H, xsg);
    constexpr int NROWS = R == 1 ? 4 : 2;   // whole units (gate and up row) per lane
    warp_rows<B, NROWS, R>(units, rowb, 2 * cnt, H, xq, xsg, [&](int rb, const float (&acc)[NROWS][R]) {
#pragma unroll
        for (int k2 = 0; k2 < NROWS; k2 += 2) {
            if (rb + k2 + 1 < 2 * cnt) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (r < nv) {
                        const float gt = acc[k2][r], up = acc[k2 + 1][r];
                        const uint32_t a = __float_as_uint(gt / (1.0f + expf(-gt)) * up);
#pragma unroll
                        for (int c = 0; c < kActCopies; ++c)
                            st_tag(dst + c * cs + (size_t)rows[r] * ld + ((rb + k2) >> 1), a, tag);
                    }
            }
        }
    });
}

// Stores v at element i of dst: a plain fp32 array, or (tag != 0) tagged words.
__device__ __forceinline__ void put_out(void *dst, size_t i, float v, unsigned tag)
{
    if (tag) st_tag(static_cast<uint64_t *>(dst) + i, __float_as_uint(v), tag);
    else static_cast<float *>(dst)[i] = v;
}

// Down rows [0, cnt) (K inputs each) against the staged activation pairs
// pair0 + t, t = g0 .. (t < popc(mask)): dst[h * hs + t * ts] (see put_out).
template <int B, int R>
__device__ __forceinline__ void dn_k_body(const float4 *act, const float *asum, int K, const uint8_t *rows0, int cnt,
                                  int rowb, uint32_t mask, int pair0, int g0, void *dst, int hs, int ts, unsigned tag)
{
    const int Gi = K / kGroup, n = __popc(mask);
    int tp[R];
    int nv = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        tp[r] = g0 + r < n ? g0 + r : n - 1;
        nv += g0 + r < n ? 1 : 0;
    }
    uint32_t xq[R];
    int soff[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        xq[r] = smem_u32(act) + (uint32_t)((pair0 + tp[r]) * K * 4);
        soff[r] = (pair0 + tp[r]) * Gi;
    }
    float xsg[R][kMaxGPL];
    lane_gsums<R>(smem_u32(asum), soff, K, xsg);
    constexpr int NROWS = R == 1 ? 2 : 1;   // (down rows: any count)
    warp_rows<B, NROWS, R>(rows0, rowb, cnt, K, xq, xsg, [&](int rb, const float (&acc)[NROWS][R]) {
#pragma unroll
        for (int k2 = 0; k2 < NROWS; ++k2)
            if (rb + k2 < cnt) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    if (r < nv) put_out(dst, (size_t)(rb + k2) * hs + (size_t)tp[r] * ts, acc[k2][r], tag);
            }
    });
}

// Out-of-line entry points of the row kernels (one per instantiation).
template <int B, int R>
__device__ __noinline__ void gu_k(const float4 *xs, const float *xsum, int H, const uint8_t *units, int cnt,
                                  int rowb, uint32_t mask, int g0, uint64_t *dst, int ld, size_t cs, unsigned tag)
{
    gu_k_body<B, R>(xs, xsum, H, units, cnt, rowb, mask, g0, dst, ld, cs, tag);
}
template <int B, int R>
__device__ __noinline__ void dn_k(const float4 *act, const float *asum, int K, const uint8_t *rows0, int cnt,
                                  int rowb, uint32_t mask, int pair0, int g0, void *dst, int hs, int ts, unsigned tag)
{
    dn_k_body<B, R>(act, asum, K, rows0, cnt, rowb, mask, pair0, g0, dst, hs, ts, tag);
}

// ---------------------------------------------- one token vector in registers
//
// When a call has one token vector (one row of the mask) and a row has at
// most 32 groups (K <= 2048), each lane of a row keeps its group's 64 inputs
// in registers and the warp walks the rows: per row only the codes, scale and
// bias are read from shared memory, and the loop body is small enough to run
// from the innermost instruction cache after the first row.  The arithmetic
// per row is that of grp_cls with NR = 1 (same sub-group visit order, same
// class accumulators, same lane reduction), so a row's result is bit-for-bit
// the one the general kernels give.

// Sub-group of group g visited at position v (0 .. 3) by for_subgroups.
template <int BITS>
__device__ __forceinline__ int visit_sg(int g, int v)
{
    if constexpr (BITS == 6) return 2 * ((v >> 1) ^ ((g >> 3) & 1)) + (v & 1);
    else if constexpr (BITS == 8) return (v + chunk_rot<8>(g)) & 3;
    else return 2 * (((v >> 1) + chunk_rot<4>(g)) & 1) + (v & 1);
}

// The lane's inputs of group g of an arranged vector at shared address xq,
// in visit order: x[4 v + t] = inputs 64 g + 4 (4 sg + t) .., sg = visit_sg(g, v).
template <int BITS>
__device__ __forceinline__ void load_x1(uint32_t xq, int g, int G, float4 (&x)[16])
{
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int sg = visit_sg<BITS>(g, v);
#pragma unroll
        for (int t = 0; t < 4; ++t) x[4 * v + t] = ldsf4(xq + g * 16 + (4 * sg + t) * G * 16);
    }
}

// The lane's part of row . x (group g), before the reduction over the lanes
// of the row: exactly grp_cls<BITS, 1, 1> on a zero accumulator.
template <int BITS>
__device__ __forceinline__ float dot1(uint32_t row, int g, int K, const float4 (&x)[16], float xsum)
{
    using PT = Pairs<BITS>;
    constexpr int NC = PT::NC, NA = BITS == 6 ? NC : 2 * NC;
    float s, b;
    scale_bias(row, K, BITS, g, s, b);
    float2 A[NA];
#pragma unroll
    for (int c = 0; c < NA; ++c) A[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int sg = visit_sg<BITS>(g, v);
        uint32_t w[BITS / 2];
        if constexpr (BITS == 6) {
            // 12 bytes at row + 48 g + 12 sg: 8-byte aligned for even sg
            const uint32_t a = row + g * 48 + 12 * sg;
            if (sg & 1) {
                w[0] = lds1(a);
                const uint2 p = lds2(a + 4);
                w[1] = p.x; w[2] = p.y;
            } else {
                const uint2 p = lds2(a);
                w[0] = p.x; w[1] = p.y;
                w[2] = lds1(a + 8);
            }
        } else if constexpr (BITS == 8) {
            const uint4 p = lds4(row + g * 64 + 16 * sg);
            w[0] = p.x; w[1] = p.y; w[2] = p.z; w[3] = p.w;
        } else {
            const uint2 p = lds2(row + g * 32 + 8 * sg);
            w[0] = p.x; w[1] = p.y;
        }
        const int half = NA > NC ? (v & 1) * NC : 0;
        PT::each(w, [&](int i, float a, float bb) {
            A[PT::cls(i) + half] = __ffma2_rn(make_float2(a, bb), xpair(x[4 * v + (i >> 1)], i & 1), A[PT::cls(i) + half]);
        });
    }
    float t = 0.f;
#pragma unroll
    for (int c = 0; c < NA; ++c) {
        const int i0 = first_of_class<PT>(c % NC);
        t = fmaf(A[c].x, __uint_as_float(cls_bits(PT::pa(i0))), t);
        t = fmaf(A[c].y, __uint_as_float(cls_bits(PT::pb(i0))), t);
    }
    return fmaf(s, t, fmaf(b, xsum, 0.f));
}

// Rows against one token vector: the warp takes rows r0 + RPP i (lanes
// lg of a row group, RPP = 32 / LPR row groups) of nrows at rows + r * rstride
// (shared memory), each of K inputs.  emit(r, value) runs on the first lane
// of the row group with the complete dot product of row r.
template <int BITS, typename F>
__device__ __forceinline__ void rows1(uint32_t rows, int rstride, int nrows, int K, uint32_t xq, uint32_t xsq, F &&emit)
{
    const int lane = threadIdx.x & 31;
    const int G = K >> 6, lgL = ilog2(G), LPR = 1 << lgL, RPP = 32 >> lgL;
    const int g = lane & (LPR - 1), lr = lane >> lgL;
    float4 x[16];
    load_x1<BITS>(xq, g, G, x);
    const float xsum = ldsf1(xsq + 4 * g);
#pragma unroll 1
    for (int r0 = 0; r0 < nrows; r0 += RPP) {
        const int r = r0 + lr;
        float acc = dot1<BITS>(rows + (uint32_t)(min(r, nrows - 1) * rstride), g, K, x, xsum);
#pragma unroll 1
        for (int o = LPR >> 1; o >= 1; o >>= 1) acc += __shfl_xor_sync(FULLMASK, acc, o);
        if (g == 0 && r < nrows) emit(r, acc);
    }
}

// Gate/up units [0, cnt) (unit u: gate row 2u, up row 2u + 1) against one
// token vector: dst[u] = silu(gate) * up, tagged.  A row group takes a whole
// unit.
template <int BITS>
__device__ __noinline__ void gu1(uint32_t units, int cnt, int rowb, int H, uint32_t xq, uint32_t xsq, uint64_t *dst,
                                 size_t cs, unsigned tag)
{
    const int lane = threadIdx.x & 31;
    const int G = H >> 6, lgL = ilog2(G), LPR = 1 << lgL, RPP = 32 >> lgL;
    const int g = lane & (LPR - 1), lr = lane >> lgL;
    float4 x[16];
    load_x1<BITS>(xq, g, G, x);
    const float xsum = ldsf1(xsq + 4 * g);
#pragma unroll 1
    for (int u0 = 0; u0 < cnt; u0 += RPP) {
        const uint32_t ru = units + (uint32_t)(2 * min(u0 + lr, cnt - 1) * rowb);
        float gt = 0.f, up = 0.f;
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
            const float v = dot1<BITS>(ru + k * rowb, g, H, x, xsum);
            if (k) up = v;
            else gt = v;
        }
#pragma unroll 1
        for (int o = LPR >> 1; o >= 1; o >>= 1) {
            gt += __shfl_xor_sync(FULLMASK, gt, o);
            up += __shfl_xor_sync(FULLMASK, up, o);
        }
        if (g == 0 && u0 + lr < cnt) {
            const uint32_t a = __float_as_uint(gt / (1.0f + expf(-gt)) * up);
#pragma unroll
            for (int c = 0; c < kActCopies; ++c) st_tag(dst + c * cs + u0 + lr, a, tag);
        }
    }
}

// Rows [0, cnt) against one vector: dst[r * ds] = row r . x (see put_out).
template <int BITS>
__device__ __noinline__ void plain1(uint32_t rows, int cnt, int rowb, int K, uint32_t xq, uint32_t xsq, void *dst, int ds,
                                    unsigned tag)
{
    rows1<BITS>(rows, rowb, cnt, K, xq, xsq, [&](int r, float v) { put_out(dst, (size_t)r * ds, v, tag); });
}

// Dispatch on (bits, row-group size): code = bits * 8 + nr.
#define MOE_RK_CASES(FN, ARGS)                                                                   \
    case 4 * 8 + 1: FN<4, 1> ARGS; break;                                                        \
    case 4 * 8 + 2: FN<4, 2> ARGS; break;                                                        \
    case 6 * 8 + 1: FN<6, 1> ARGS; break;                                                        \
    case 6 * 8 + 2: FN<6, 2> ARGS; break;                                                        \
    case 8 * 8 + 1: FN<8, 1> ARGS; break;                                                        \
    case 8 * 8 + 2: FN<8, 2> ARGS; break;

__device__ __noinline__ void gu_units(const Sh &sh, int H, int bits, const uint8_t *units, int cnt, int rowb,
                                         uint32_t mask, uint64_t *dst, int ld, size_t cs, unsigned tag)
{
    if (__popc(mask) == 1 && H <= 32 * kGroup && bits != 0) {
        const int m = __ffs(mask) - 1;
        const uint32_t xq = smem_u32(sh.xs) + (uint32_t)(m * H * 4), xsq = smem_u32(sh.xsum) + (uint32_t)(m * (H / kGroup) * 4);
        uint64_t *d = dst + (size_t)m * ld;
        if (bits == 6) gu1<6>(smem_u32(units), cnt, rowb, H, xq, xsq, d, cs, tag);
        else if (bits == 8) gu1<8>(smem_u32(units), cnt, rowb, H, xq, xsq, d, cs, tag);
        else gu1<4>(smem_u32(units), cnt, rowb, H, xq, xsq, d, cs, tag);
        return;
    }
    for_row_groups(mask, [&](int g0, int nr) {
        switch (bits * 8 + nr) {
            MOE_RK_CASES(gu_k, (sh.xs, sh.xsum, H, units, cnt, rowb, mask, g0, dst, ld, cs, tag))
        default: break;
        }
    });
}

// dst[h * hs + t * ts] for down row h and the staged pair pair0 + t (t the
// rank of a row in `mask`): plain fp32, or tagged words when tag != 0.
__device__ __noinline__ void dn_rows(const Sh &sh, int bits, const uint8_t *rows0, int cnt, int rowb, int K,
                                        uint32_t mask, int pair0, void *dst, int hs, int ts, unsigned tag)
{
    if (__popc(mask) == 1 && K <= 32 * kGroup && bits != 0) {
        const uint32_t xq = smem_u32(sh.act) + (uint32_t)(pair0 * K * 4), xsq = smem_u32(sh.asum) + (uint32_t)(pair0 * (K / kGroup) * 4);
        if (bits == 6) plain1<6>(smem_u32(rows0), cnt, rowb, K, xq, xsq, dst, hs, tag);
        else if (bits == 8) plain1<8>(smem_u32(rows0), cnt, rowb, K, xq, xsq, dst, hs, tag);
        else plain1<4>(smem_u32(rows0), cnt, rowb, K, xq, xsq, dst, hs, tag);
        return;
    }
    for_row_groups(mask, [&](int g0, int nr) {
        switch (bits * 8 + nr) {
            MOE_RK_CASES(dn_k, (sh.act, sh.asum, K, rows0, cnt, rowb, mask, pair0, g0, dst, hs, ts, tag))
        default: break;
        }
    });
}

// ------------------------------------------------------------ P0: RMSNorm

// hn rows of x (bf16 [M, H], global) -> xs (arranged, * 2^100) and group
// sums; 1 / rms of row m -> red[m * kRed + kSsChunks].  A thread item is 8
// consecutive inputs (one 16-byte load); H / 8 is a multiple of 32, so the
// 32 items of a warp are one aligned chunk of 256 inputs of one row.  The
// sum of squares is the chunks' warp sums added in chunk order: the same
// for every row whatever M is and however many warps take part.  Run by compute warps w0 .. NCW - 1
// (the first w0 route meanwhile), which meet at their own named barrier.
__device__ void build_hn(const KParams &kp, const Sh &sh, const void *x, unsigned xtag, const uint16_t *gamma,
                         int w0)
{
    const int H = kp.g.H, M = kp.M, G = H / kGroup, lane = threadIdx.x & 31;
    const int tid = threadIdx.x - 32 * w0, nt = 32 * (NCW - w0);
    const int per_row = H / 8, lpr = ilog2(per_row), total = M * per_row;
    auto bar = [nt]() { asm volatile("bar.sync 5, %0;" ::"r"(nt) : "memory"); };
    // pass 1: sums of squares per (row, warp); raw values into xs.  Several
    // items per thread and round, all loads in flight before any is used.
    auto item = [&](int it, const uint32_t (&aw)[4]) {
        float ss = 0.f;
        if (it < total) {
            const int m = it >> lpr, c = it & (per_row - 1);
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = __uint_as_float(aw[j] << 16);
                f[2 * j + 1] = __uint_as_float(aw[j] & 0xFFFF0000u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
            // inputs 8c .. 8c+7: group c / 8, quads 2 (c % 8) and 2 (c % 8) + 1
            const int g = c >> 3, t = (c & 7) * 2;
            float4 *row = sh.xs + (size_t)m * (H / 4);
            row[t * G + g] = make_float4(f[0], f[1], f[2], f[3]);
            row[(t + 1) * G + g] = make_float4(f[4], f[5], f[6], f[7]);
        }
        ss = warp_sum(ss);
        const int wfirst = it - lane;
        if (lane == 0 && wfirst < total) sh.red[(wfirst >> lpr) * kRed + ((wfirst & (per_row - 1)) >> 5)] = ss;
    };
    constexpr int NI = 4;   // items per thread and round
#pragma unroll 1
    for (int base = 0; base < total; base += NI * nt) {
        uint32_t a[NI][4];
        if (xtag) {
            // the previous layer's output: tagged bf16 pairs
            const uint64_t *xt = static_cast<const uint64_t *>(x);
            const uint64_t *p[NI];
#pragma unroll
            for (int n = 0; n < NI; ++n) {
                const int it = base + tid + n * nt;
                p[n] = it < total ? xt + (size_t)(it >> lpr) * (H / 2) + 4 * (it & (per_row - 1)) : nullptr;
            }
            poll_items<NI>(sh, p, xtag, 40, a);
        } else {
            const uint4 *xp = reinterpret_cast<const uint4 *>(x);
#pragma unroll
            for (int n = 0; n < NI; ++n) {
                const int it = base + tid + n * nt;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (it < total) v = __ldcg(xp + it);
                a[n][0] = v.x; a[n][1] = v.y; a[n][2] = v.z; a[n][3] = v.w;
            }
        }
#pragma unroll
        for (int n = 0; n < NI; ++n)
            if (n == 0 || base + n * nt < total) item(base + tid + n * nt, a[n]);
    }
    bar();
    if (tid == 0 && xtag) stamp(kp, (int)(xtag - sh.epoch), 16);
    if (tid < M) {
        float t = 0.f;
#pragma unroll 1
        for (int c = 0; c < per_row / 32; ++c) t += sh.red[tid * kRed + c];
        sh.red[tid * kRed + kSsChunks] = rsqrtf(t / (float)H + kp.g.eps);
    }
    bar();
    if (tid == 0 && xtag) stamp(kp, (int)(xtag - sh.epoch), 20);
    // pass 2: scale by rinv * gamma * 2^100, and the group sums of hn (8
    // consecutive items make a group)
#pragma unroll 1
    for (int base = 0; base < total; base += nt) {
        const int it = base + tid;
        float gs = 0.f;
        if (it < total) {
            const int m = it >> lpr, c = it & (per_row - 1);
            const float rinv = sh.red[m * kRed + kSsChunks];
            const uint4 gv = *reinterpret_cast<const uint4 *>(gamma + c * 8);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            const int g = c >> 3, t = (c & 7) * 2;
            float4 *row = sh.xs + (size_t)m * (H / 4);
            const float4 a = row[t * G + g], b = row[(t + 1) * G + g];
            float h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                h[2 * j] = h[2 * j] * rinv * __uint_as_float(gw[j] << 16);
                h[2 * j + 1] = h[2 * j + 1] * rinv * __uint_as_float(gw[j] & 0xFFFF0000u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) gs += h[j];
            row[t * G + g] = make_float4(h[0] * kXScale, h[1] * kXScale, h[2] * kXScale, h[3] * kXScale);
            row[(t + 1) * G + g] = make_float4(h[4] * kXScale, h[5] * kXScale, h[6] * kXScale, h[7] * kXScale);
        }
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) gs += __shfl_xor_sync(FULLMASK, gs, o);
        if (it < total && (it & 7) == 0) {
            const int m = it >> lpr, c = it & (per_row - 1);
            sh.xsum[m * G + (c >> 3)] = gs;
        }
    }
    if (tid == 0 && xtag) stamp(kp, (int)(xtag - sh.epoch), 21);
    bar();
}

// Partial router dots (every compute warp, at the start of a layer): the
// CTA dots every router row with gamma * x over its own output slice of the
// layer input, and adds up x^2 over the slice, for each token row m, and
// publishes the Er + 1 sums as tagged words part[m][e][CTA] (e = Er: the
// squares).  The logit of router row e is rinv_m times the sum over CTAs of
// part[m][e][.], rinv_m = 1 / sqrt(sum over CTAs of part[m][Er][.] / H +
// eps) (reduce_logits sums, top-k scales): the RMSNorm's scale is a common
// factor of the row's products (flash-moe, "Metal Compute Shaders": RMS
// normalisation; PureDrive model card, "Summary": the router of 256 experts
// plus the shared expert's gate), so no CTA needs the whole input first.
// The slice of x is the CTA's own output of the previous layer, which
// combine left in shared memory (layer 0: the caller's rows).  Quantised
// rows: each weight dequantised as s q + b (fp32) before its product.
__device__ void router_partials(const KParams &kp, const Sh &sh, const uint64_t *part, int l)
{
    const Geo &g = kp.g;
    const CtaPlan &b = *sh.cp;
    const int M = kp.M, H = g.H, nh = b.nh, h0 = b.h0, Er = g.Er, E1 = Er + 1, Erp = g.Erp, P = gridDim.x;
    const int hr = sh.hrows, tid = threadIdx.x;
    const unsigned tag = layer_tag(sh, l);
    const uint16_t *gamma = reinterpret_cast<const uint16_t *>(sh.pb);
    float *u = sh.ru, *xv = sh.ru + kMaxRows * hr;
#pragma unroll 1
    for (int t = tid; t < M * nh; t += NCT) {
        const int m = t / nh, j = t - m * nh;
        if (l == 0) xv[m * hr + j] = bf2f(kp.x[(size_t)m * H + h0 + j]);
        u[m * hr + j] = xv[m * hr + j] * bf2f(gamma[h0 + j]);
    }
    cbar();
    if (tid == 0) stamp(kp, l, 17);
    const uint8_t *codes = sh.pb + b.off_router;
    const uint32_t *sbw = reinterpret_cast<const uint32_t *>(sh.pb + b.off_rsb);
    const float *wf = reinterpret_cast<const float *>(sh.pb + b.off_router);
    // columns from js on belong to the slice's second group
    const int js = b.ng > 1 ? (b.g0 + 1) * kGroup - h0 : nh;
    uint64_t *dst = const_cast<uint64_t *>(part) + blockIdx.x;
    // items rotated by the routing warps' threads, so that items past the
    // first NCT go to the other warps and the routing warps start reducing
    // first
    const int rot = (tid + 32 * M) % NCT;
#pragma unroll 1
    for (int t = rot; t < M * E1; t += NCT) {
        const int m = t / E1, e = t - m * E1;
        const float *um = u + m * hr;
        float acc = 0.f;
        if (e == Er) {
            const float *xm = xv + m * hr;
#pragma unroll 4
            for (int j = 0; j < nh; ++j) acc = fmaf(xm[j], xm[j], acc);
        } else if (g.qb) {
            const uint32_t w0 = sbw[e], w1 = b.ng > 1 ? sbw[Erp + e] : w0;
            const float s0 = __uint_as_float(w0 << 16), b0 = __uint_as_float(w0 & 0xFFFF0000u);
            const float s1 = __uint_as_float(w1 << 16), b1 = __uint_as_float(w1 & 0xFFFF0000u);
#pragma unroll 4
            for (int j = 0; j < nh; ++j) {
                const bool hi = j >= js;
                const float wt = fmaf(hi ? s1 : s0, code_float(codes[j * Erp + e]), hi ? b1 : b0);
                acc = fmaf(wt, um[j], acc);
            }
        } else {
#pragma unroll 4
            for (int j = 0; j < nh; ++j) acc = fmaf(wf[j * Erp + e], um[j], acc);
        }
        st_tag(dst + (size_t)t * P, __float_as_uint(acc), tag);
    }
}

// The logits of this CTA's router rows [ra, rb) for token row m, before
// the RMSNorm scale, or (row Er) the row's sum of squares (one warp): every
// CTA's partial sums, each lane adding
// CTAs lane, lane + 32, ... in turn and the lanes then combined by a
// butterfly (every lane ends with the same sums; the order depends on
// nothing but the row), published as tagged words, kLogitCopies copies
// each.  The words of a router row are read by this CTA alone.
__device__ __noinline__ void reduce_logits(const KParams &kp, const Sh &sh, const uint64_t *part, uint64_t *logits,
                                           int m, int l)
{
    const Geo &g = kp.g;
    const CtaPlan &b = *sh.cp;
    const int lane = threadIdx.x & 31, E1 = g.Er + 1, nr = b.rb - b.ra, P = gridDim.x;
    const unsigned tag = layer_tag(sh, l);
    if (nr <= 0) return;
    constexpr int NC = (kMaxCtas + 31) / 32;
    const uint64_t *rows = part + ((size_t)m * E1 + b.ra) * P;
    // all words of the lane's CTAs requested together, then every missing
    // one again in each round until all are there (each word has this one
    // reader); the rounds are the whole warp's, so that no lane's wait is
    // serialised behind another's (bounded: zeros after a timeout)
    uint64_t v[NC][kRouterRowsCta];
#pragma unroll
    for (int i = 0; i < NC; ++i)
#pragma unroll
        for (int r = 0; r < kRouterRowsCta; ++r) {
            const int c = lane + 32 * i;
            v[i][r] = c < P && r < nr ? ld_tag(rows + (size_t)r * P + c) : (uint64_t)tag << 32;
        }
    unsigned long long t0 = 0;
    unsigned it = 0;
#pragma unroll 1
    for (;;) {
        bool missing = false;
#pragma unroll
        for (int i = 0; i < NC; ++i)
#pragma unroll
            for (int r = 0; r < kRouterRowsCta; ++r) missing |= (unsigned)(v[i][r] >> 32) != tag;
        if (!__any_sync(FULLMASK, missing)) break;
        if (!__all_sync(FULLMASK, poll_more(sh, ++it, t0, 45))) {
#pragma unroll
            for (int i = 0; i < NC; ++i)
#pragma unroll
                for (int r = 0; r < kRouterRowsCta; ++r) v[i][r] = (uint64_t)tag << 32;
            break;
        }
#pragma unroll
        for (int i = 0; i < NC; ++i)
#pragma unroll
            for (int r = 0; r < kRouterRowsCta; ++r)
                if ((unsigned)(v[i][r] >> 32) != tag) v[i][r] = ld_tag(rows + (size_t)r * P + lane + 32 * i);
    }
    if (threadIdx.x == 0) stamp(kp, l, 23);
    float acc[kRouterRowsCta];
#pragma unroll
    for (int r = 0; r < kRouterRowsCta; ++r) {
        acc[r] = 0.f;
#pragma unroll
        for (int i = 0; i < NC; ++i)
            if (lane + 32 * i < P && r < nr) acc[r] += __uint_as_float((uint32_t)v[i][r]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int r = 0; r < kRouterRowsCta; ++r) acc[r] += __shfl_xor_sync(FULLMASK, acc[r], o);
#pragma unroll
    for (int r = 0; r < kRouterRowsCta; ++r) {
        const int e = b.ra + r;
        // (debug switch: one logit of layer 0 stays unpublished)
        if (r < nr && lane < kLogitCopies && !(l == 0 && kp.skip_row == e))
            st_tag(logits + ((size_t)lane * kp.ws_l.maxr + m) * E1 + e, __float_as_uint(acc[r]), tag);
    }
}

// Activations (fp32 rows in global memory) of `n` staged pairs: pair p =
// src(p)[0 .. K), arranged, * 2^100, with group sums.  A thread item is 4
// consecutive inputs; 16 items make a group.
// nt threads of whole compute warps take part, the calling one as number tid.  The
// sources are tagged fp32 words; each is waited for until it carries `tag`.
template <typename F>
__device__ __forceinline__ void stage_acts(const Sh &sh, int n, int K, int tid, int nt, unsigned tag, F &&src)
{
    const int per = K / 4, lgp = ilog2(per), G = K / kGroup, total = n * per;
    // an item's 4 inputs into the staging buffer; returns their sum
    auto item = [&](int it, const uint32_t (&u)[4]) -> float {
        float gs = 0.f;
        if (it < total) {
            const int p = it >> lgp, c = it & (per - 1);
            const float4 v = make_float4(__uint_as_float(u[0]), __uint_as_float(u[1]), __uint_as_float(u[2]),
                                         __uint_as_float(u[3]));
            gs = (v.x + v.y) + (v.z + v.w);
            sh.act[(size_t)p * per + (c & 15) * G + (c >> 4)] =
                make_float4(v.x * kXScale, v.y * kXScale, v.z * kXScale, v.w * kXScale);
        }
        return gs;
    };
    // four items per thread and round, all loads in flight before any is used
    constexpr int NI = 4;
#pragma unroll 1
    for (int base = 0; base < total; base += NI * nt) {
        const uint64_t *p[NI];
#pragma unroll
        for (int n = 0; n < NI; ++n) {
            const int it = base + tid + n * nt;
            p[n] = it < total ? src(it >> lgp) + 4 * (it & (per - 1)) : nullptr;
        }
        uint32_t a[NI][4];
        poll_items<NI>(sh, p, tag, 41, a);
        // group sums (16 consecutive items make a group), the items'
        // reductions interleaved
        float gs[NI];
#pragma unroll
        for (int n = 0; n < NI; ++n) gs[n] = item(base + tid + n * nt, a[n]);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
            for (int n = 0; n < NI; ++n) gs[n] += __shfl_xor_sync(FULLMASK, gs[n], o);
#pragma unroll
        for (int n = 0; n < NI; ++n) {
            const int it = base + tid + n * nt;
            if (it < total && (it & 15) == 0) sh.asum[(it >> lgp) * G + ((it & (per - 1)) >> 4)] = gs[n];
        }
    }
}

// ------------------------------------------------------------- R: routing

// Order-preserving map of a float to an unsigned key (larger float, larger
// key) and back.
__device__ __forceinline__ uint32_t fkey(float v)
{
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unkey(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k of router row m by one warp, keyed on (logit descending, expert id
// ascending); lane `lane` holds experts lane + 32 i.  k rounds: the warp-wide
// largest of the lanes' best remaining keys (redux.sync); the lane holding
// it at its lowest index drops it and records it.  Exact ties between lanes
// (several lanes hold the largest key) go to the lowest expert id.
// Writes topv/tope/topw (selection order), row_w/row_pair (expert-id order;
// row_pair holds the expert id until the slot table is built) and sigma.
template <int NPL>
__device__ __noinline__ void topk_row_t(const KParams &kp, const Sh &sh, int m, const uint64_t *logits, unsigned tag)
{
    const int lane = threadIdx.x & 31;
    const int E = kp.g.E, k = kp.g.k, Er = kp.g.Er;
    // this CTA's copy of the logits
    const uint64_t *row = logits + ((size_t)(blockIdx.x % kLogitCopies) * kp.ws_l.maxr + m) * (Er + 1);
    // the lane's logits, the shared expert's gate logit and the row's sum of
    // squares, all loaded together, then in each round of the whole warp
    // every word still missing again
    const uint64_t none = (uint64_t)tag << 32;
    uint64_t v[NPL + 2];
    auto addr = [&](int i) { return i < NPL ? row + lane + 32 * i : i == NPL ? row + E : row + Er; };
#pragma unroll
    for (int i = 0; i < NPL; ++i) v[i] = lane + 32 * i < E ? ld_tag(addr(i)) : none;
    v[NPL] = kp.g.has_shared ? ld_tag(addr(NPL)) : none;
    v[NPL + 1] = ld_tag(addr(NPL + 1));
    unsigned long long t0 = 0;
    unsigned it = 0;
#pragma unroll 1
    for (;;) {
        bool missing = false;
#pragma unroll
        for (int i = 0; i < NPL + 2; ++i) missing |= (unsigned)(v[i] >> 32) != tag;
        if (!__any_sync(FULLMASK, missing)) break;
        if (!__all_sync(FULLMASK, poll_more(sh, ++it, t0, 42))) break;
#pragma unroll
        for (int i = 0; i < NPL + 2; ++i)
            if ((unsigned)(v[i] >> 32) != tag) v[i] = ld_tag(addr(i));
    }
    if (threadIdx.x == 0) stamp(kp, (int)(tag - sh.epoch - 1u), 15);
    uint32_t key[NPL];
    // the published logits are the router dots before the RMSNorm scale
    const float rinv = rsqrtf(__uint_as_float((uint32_t)v[NPL + 1]) / (float)kp.g.H + kp.g.eps);
#pragma unroll
    for (int i = 0; i < NPL; ++i)
        key[i] = lane + 32 * i < E ? fkey(__uint_as_float((uint32_t)v[i]) * rinv) : 0u;
    const float lsg = __uint_as_float((uint32_t)v[NPL]) * rinv;
    float *topv = sh.topv + m * kMaxK;
    int *tope = sh.tope + m * kMaxK;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        uint32_t t[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) t[i] = key[i];
#pragma unroll
        for (int w = NPL >> 1; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) t[i] = max(t[i], t[i + w]);
        const uint32_t wk = __reduce_max_sync(FULLMASK, t[0]);
        // the lane's lowest index holding wk (NPL if none)
        int bi = NPL;
#pragma unroll
        for (int i = NPL - 1; i >= 0; --i) bi = key[i] == wk ? i : bi;
        const unsigned bal = __ballot_sync(FULLMASK, bi < NPL);
        int wl = __ffs(bal) - 1;
        if (bal & (bal - 1u)) {
            const unsigned we = __reduce_min_sync(FULLMASK, bi < NPL ? (unsigned)(lane + 32 * bi) : 0xFFFFFFFFu);
            wl = (int)(we & 31u);
        }
        if (lane == wl) {
#pragma unroll
            for (int i = 0; i < NPL; ++i) key[i] = i == bi ? 0u : key[i];
            topv[r] = unkey(wk);
            tope[r] = lane + 32 * bi;
        }
    }
    __syncwarp();
#ifdef MOE_DEBUG_BOUNDS
    // test hook of the checked build: row 0 of the first layer reports the
    // id set by moe_debug_inject as its first choice
    if (kp.inject_e >= 0 && tag == layer_tag(sh, 0) && m == 0 && lane == 0) tope[0] = kp.inject_e;
    __syncwarp();
#endif
    // renormalised softmax weights over the k kept logits (the full softmax
    // probabilities divided by their top-k sum)
    const float ev = lane < k ? expf(topv[lane] - topv[0]) : 0.f;
    const float z = warp_sum(ev);
    if (lane < k) {
        const float wv = ev / z;
        const int e = tope[lane];
        int r = 0;
#pragma unroll 1
        for (int j = 0; j < k; ++j) r += tope[j] < e ? 1 : 0;
        sh.topw[m * kMaxK + lane] = wv;
        sh.row_w[m * kMaxK + r] = wv;
        sh.row_pair[m * kMaxK + r] = e;
    }
    if (lane == 0) sh.sigma[m] = kp.g.has_shared ? 1.0f / (1.0f + expf(-lsg)) : 0.f;
}

__device__ void topk_row(const KParams &kp, const Sh &sh, int m, const uint64_t *logits, unsigned tag)
{
    const int E = kp.g.E;
    if (E <= 64) topk_row_t<2>(kp, sh, m, logits, tag);
    else if (E <= 256) topk_row_t<8>(kp, sh, m, logits, tag);
    else topk_row_t<16>(kp, sh, m, logits, tag);
}

// Named barrier over the first nw compute warps (the routing warps).
__device__ __forceinline__ void rbar(int nw) { asm volatile("bar.sync 2, %0;" ::"r"(nw * 32) : "memory"); }

// Routing, run by the first M compute warps only (one per token row); the
// other warps work meanwhile.  Builds the slot table (the distinct experts
// of the M rows in id order, each with the mask of rows that chose it and
// the index of its first activation pair) and turns row_pair into pair
// indices; ends by telling the producer that the table of layer l is ready.
__device__ void route(const KParams &kp, const Sh &sh, const uint64_t *logits, int l)
{
    const unsigned tag = layer_tag(sh, l);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = kp.g.E, k = kp.g.k, M = kp.M;
    if (M > 1 && warp == 0) {
#pragma unroll 1
        for (int e = lane; e < E; e += 32) sh.emask[e] = 0u;
    }
    topk_row(kp, sh, warp, logits, tag);
    if (threadIdx.x == 0) stamp(kp, l, 12);
    if (M > 1) rbar(M);
    if (warp != 0) return;
    int U, npairs;
    if (M == 1) {
        // one row: the slots are its k experts in id order
#pragma unroll 1
        for (int j = lane; j < k; j += 32) {
            sh.slot_e[j] = chk(sh, sh.row_pair[j], E, 1);
            sh.slot_mask[j] = 1u;
            sh.slot_rowbase[j] = j;
            sh.row_pair[j] = j;
        }
        U = npairs = k;
    } else {
#pragma unroll 1
        for (int m = 0; m < M; ++m)
#pragma unroll 1
            for (int j = lane; j < k; j += 32) atomicOr(&sh.emask[chk(sh, sh.tope[m * kMaxK + j], E, 2)], 1u << m);
        __syncwarp();
        U = 0;
#pragma unroll 1
        for (int c0 = 0; c0 < E; c0 += 32) {
            const int e = c0 + lane;
            const uint32_t em = e < E ? sh.emask[e] : 0u;
            const unsigned bal = __ballot_sync(FULLMASK, em != 0u);
            if (em) {
                const int pos = chk(sh, U + __popc(bal & ((1u << lane) - 1u)), kp.ws_l.max_slots, 3);
                sh.slot_e[pos] = e;
                sh.slot_mask[pos] = em;
                sh.eslot[e] = pos;
            }
            U += __popc(bal);
        }
        U = min(U, kp.ws_l.max_slots);
        __syncwarp();
        // pair bases: prefix sums of popc(mask) over the slots
        npairs = 0;
#pragma unroll 1
        for (int s0 = 0; s0 < U; s0 += 32) {
            const int s = s0 + lane;
            const int pc = s < U ? __popc(sh.slot_mask[s]) : 0;
            int inc = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULLMASK, inc, o);
                if (lane >= o) inc += t;
            }
            if (s < U) sh.slot_rowbase[s] = npairs + inc - pc;
            npairs += __shfl_sync(FULLMASK, inc, 31);
        }
        __syncwarp();
#pragma unroll 1
        for (int m = 0; m < M; ++m)
#pragma unroll 1
            for (int j = lane; j < k; j += 32) {
                const int s = chk(sh, sh.eslot[chk(sh, sh.row_pair[m * kMaxK + j], E, 4)], U, 5);
                sh.row_pair[m * kMaxK + j] = sh.slot_rowbase[s] + __popc(sh.slot_mask[s] & ((1u << m) - 1u));
            }
    }
    // a streamed layer's experts are read from its HBM cache: the slot table
    // carries their cache slots in place of their ids (the ids keep ordering
    // the combine through row_pair); an expert with no slot is reported and
    // slot 0 read instead, so every access stays inside the cache
    const LayerPtrs &Lr = kp.layer[l];
    if (Lr.slot_of && kp.mode == kModeLayers) {
#pragma unroll 1
        for (int s = lane; s < U; s += 32) {
            int c = __ldg(Lr.slot_of + sh.slot_e[s]);
            if ((unsigned)c >= (unsigned)Lr.n_slots) {
                atomicOr(&sh.ctrl->status, kStatusNotResident);
                c = 0;
            }
            sh.slot_e[s] = c;
        }
        __syncwarp();
    }
    if (kp.mode == kModeRouter && blockIdx.x == 0) {
#pragma unroll 1
        for (int m = 0; m < M; ++m)
#pragma unroll 1
            for (int j = lane; j < k; j += 32) {
                kp.idx_out[m * k + j] = sh.tope[m * kMaxK + j];
                kp.w_out[m * k + j] = sh.topw[m * kMaxK + j];
            }
    }
    if (lane == 0) {
        sh.flags[1] = U;
        sh.slot_rowbase[U] = npairs;
        stamp(kp, l, 13);
    }
    __syncwarp();
    if (lane == 0 && kp.mode == kModeLayers) mbar_arrive(sh.route, 1);
}

// ---------------------------------------------------------- workspace views

// Workspace buffers shared between CTAs, all of tagged words.
struct Ws {
    uint64_t *logits;   // [kLogitCopies][maxr][Er] fp32 (each CTA reads copy blockIdx % kLogitCopies)
    uint64_t *act;      // [kActCopies][slot][M][I] fp32 (each CTA reads copy blockIdx % kActCopies)
    uint64_t *act_s;    // [kActCopies][M][Is] fp32
    uint64_t *ping[2];  // [maxr][H / 2] bf16 pairs: layer outputs (tag of the layer that wrote them)
    uint64_t *part;     // [M][Er][CTA] fp32 partial router dots
};

__device__ __forceinline__ Ws ws_views(const KParams &kp)
{
    Ws w;
    w.logits = reinterpret_cast<uint64_t *>(kp.ws + kp.ws_l.off_logits);
    w.act = reinterpret_cast<uint64_t *>(kp.ws + kp.ws_l.off_act);
    w.act_s = reinterpret_cast<uint64_t *>(kp.ws + kp.ws_l.off_act_s);
    w.ping[0] = reinterpret_cast<uint64_t *>(kp.ws + kp.ws_l.off_ping);
    w.ping[1] = w.ping[0] + (size_t)kp.ws_l.maxr * (kp.g.H / 2);
    w.part = reinterpret_cast<uint64_t *>(kp.ws + kp.ws_l.off_part);
    return w;
}

// ------------------------------------------------------------- schedules

// This CTA's plan (run once, by one thread, into shared memory).
__device__ void cta_plan(const KParams &kp, CtaPlan &b)
{
    const Geo &g = kp.g;
    split(g.Er + 1, gridDim.x, blockIdx.x, b.ra, b.rb);
    int h1;
    hslice(g.H, b.h0, h1);
    b.nh = h1 - b.h0;
    b.ua = b.ub = 0;
    const bool sh_on = kp.mode == kModeLayers && g.has_shared;
    if (sh_on) split(g.Is, gridDim.x, blockIdx.x, b.ua, b.ub);
    b.g0 = b.h0 / kGroup;
    b.ng = b.nh > 0 ? (b.h0 + b.nh - 1) / kGroup - b.g0 + 1 : 0;
    b.off_router = (int)align_up((size_t)g.H * 2, 16);
    b.off_rsb = b.off_router + router_slice_bytes(b.nh, 0, g.Erp, g.qb);
    b.off_sdown = b.off_router + router_slice_bytes(b.nh, b.ng, g.Erp, g.qb);
    b.dpb = sh_on && b.off_sdown + b.nh * g.sd_bytes <= kp.p.pb_bytes ? b.nh : 0;
    b.off_units = b.off_sdown + b.dpb * g.sd_bytes;
    const int ub2 = 2 * g.sg_bytes;
    const int room = kp.p.pb_bytes - b.off_units;
    b.upb = ub2 > 0 ? min(b.ub - b.ua, max(0, room / ub2)) : 0;
    b.bytes = b.off_units + b.upb * ub2;
}

// Ring stages of a layer, in order: P1 units that did not fit the prefetch
// buffer, P2 routed gate/up units, P1b shared down rows that did not fit it,
// P3 routed down rows.  `f` gets (src, bytes, slot-or-kind, first, count).
// The P1 overflow is whole shared-expert units (gate row, up row); `first` is
// the unit index relative to the CTA's first shared unit.
template <typename F>
__device__ __forceinline__ void sched_p1x(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    if (kp.mode != kModeLayers || !g.has_shared || g.sg_bytes == 0) return;
    const CtaPlan &b = *sh.cp;
    const int ub2 = 2 * g.sg_bytes, cu = max(1, sh.S / ub2);
#pragma unroll 1
    for (int u = b.ua + b.upb; u < b.ub; u += cu) {
        const int n = min(cu, b.ub - u);
        f(Lp.sgu + (size_t)u * ub2, n * ub2, -2, u - b.ua, n);
    }
}

// Shared down rows that did not fit the prefetch buffer.
template <typename F>
__device__ __forceinline__ void sched_p1b(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    if (kp.mode != kModeLayers || !g.has_shared) return;
    const CtaPlan &b = *sh.cp;
    if (b.dpb) return;
    const int cd = max(1, min(sh.S / g.sd_bytes, (b.nh + 1) / 2));
#pragma unroll 1
    for (int r = 0; r < b.nh; r += cd) {
        const int n = min(cd, b.nh - r);
        f(Lp.sdown + (size_t)(b.h0 + r) * g.sd_bytes, n * g.sd_bytes, -1, r, n);
    }
}

// Expert blocks in a layer's gu / down regions: E, or a streamed layer's
// cache slots.
__device__ __forceinline__ int expert_blocks(const KParams &kp, const LayerPtrs &Lp)
{
    return Lp.slot_of ? Lp.n_slots : kp.g.E;
}

// The P2 stages of this CTA for U distinct experts: f(slot, first unit,
// units), in ring order.
template <typename F>
__device__ __forceinline__ void p2_units(const KParams &kp, const Sh &sh, int U, F &&f)
{
    const Geo &g = kp.g;
    const int ub = 2 * g.g_bytes;
    int a, b;
    split(U * g.I, gridDim.x, blockIdx.x, a, b);
    // about one stage per compute warp where the stage size allows: with one
    // token row and K <= 2048 (the one-vector kernel, a unit per pass) any
    // number of units, otherwise an even number (the general kernel's lanes
    // take two at a time)
    const bool one = kp.M == 1 && g.H <= 32 * kGroup && g.rb != 0;
    const int cu = max(1, min(sh.S / ub, one ? (b - a + NCW - 1) / NCW : 2 * ((b - a + 2 * NCW - 1) / (2 * NCW))));
    int s = (int)((unsigned)a / (unsigned)g.I), j = a - s * g.I;
#pragma unroll 1
    for (int n = a; n < b;) {
        const int cnt = min(cu, min(b - n, g.I - j));
        f(s, j, cnt);
        n += cnt;
        j += cnt;
        if (j == g.I) { j = 0; ++s; }
    }
}

template <typename F>
__device__ __forceinline__ void sched_p2(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const int ub = 2 * kp.g.g_bytes;
    p2_units(kp, sh, sh.flags[1], [&](int s, int j, int cnt) {
        f(Lp.gu + ((size_t)chk(sh, sh.slot_e[s], expert_blocks(kp, Lp), 6) * kp.g.I + j) * ub, cnt * ub, s, j, cnt);
    });
}

// P3 of this CTA: the down rows of its own output slice [h0, h0 + nh) of
// every selected expert, in slot order (one or more stages per slot).  Each
// CTA thus finishes its outputs itself (no exchange of expert outputs), and
// needs the activations of every selected expert, from every CTA.
template <typename F>
__device__ __forceinline__ void sched_p3(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, F &&f)
{
    const Geo &g = kp.g;
    const int U = sh.flags[1], h0 = sh.cp->h0, nh = sh.cp->nh;
    if (nh <= 0) return;
    const int cd = max(1, min(sh.S / g.d_bytes, nh));
#pragma unroll 1
    for (int s = 0; s < U; ++s) {
        const int e = chk(sh, sh.slot_e[s], expert_blocks(kp, Lp), 8);
#pragma unroll 1
        for (int r = 0; r < nh; r += cd) {
            const int n = min(cd, nh - r);
            f(Lp.down + ((size_t)e * g.H + h0 + r) * g.d_bytes, n * g.d_bytes, s, r, n);
        }
    }
}

// ------------------------------------------------------------- the ring

// Position of stage q in the ring: slot q % NS, phase parity (q / NS) & 1,
// and q modulo the number of consumer warps (its owner), advanced one stage
// at a time without dividing.
struct Cursor {
    int slot;
    unsigned par;
    int turn;
    bool reuse;   // the slot held an earlier stage (q >= NS)
};

__device__ __forceinline__ Cursor cursor0() { return Cursor{0, 0u, 0, false}; }

__device__ __forceinline__ void cursor_next(Cursor &c, int NS)
{
    if (++c.slot == NS) { c.slot = 0; c.par ^= 1u; c.reuse = true; }
    if (++c.turn == NCW) c.turn = 0;
}

// One batch of at most NS stages (no two in the same slot), one per lane of
// the producer warp: each lane with a stage waits until the consumer released
// the previous stage of its slot, then starts the bulk copy.  The lanes poll
// together, so the copies go out as fast as slots free up and no lane's wait
// holds up another's issue.  False on timeout or abort (the same for every
// lane).
__device__ __noinline__ bool issue_batch(const Sh &sh, bool pending, int slot, unsigned par, bool reuse,
                                         const uint8_t *src, int bytes)
{
    unsigned long long t0 = 0;
#pragma unroll 1
    for (unsigned it = 1;; ++it) {
        if (pending && (!reuse || mbar_test(&sh.empty[slot], par ^ 1u))) {
            mbar_expect_tx(&sh.full[slot], (unsigned)bytes);
            bulk_load(sh.ring + (size_t)slot * sh.S, src, (unsigned)bytes, &sh.full[slot]);
            pending = false;
        }
        if (!__any_sync(FULLMASK, pending)) return true;
        const bool go = poll_more(sh, it, t0, 1);
        if (!__all_sync(FULLMASK, go)) return false;
    }
}

// Every stage of one schedule pass (`sched` enumerates them in ring order),
// in batches of NS stages: stage base + j of a batch goes to lane j.
template <typename Sched>
__device__ __forceinline__ bool issue_pass(const Sh &sh, Cursor &c, int lane, Sched &&sched)
{
    const Cursor start = c;
#pragma unroll 1
    for (int base = 0;; base += sh.NS) {
        Cursor cur = start;
        int idx = 0;
        const uint8_t *src = nullptr;
        int bytes = 0, slot = 0;
        unsigned par = 0u;
        bool reuse = false;
        sched([&](const uint8_t *s, int b, int, int, int) {
            if (idx - base == lane && lane < sh.NS) {
                src = s;
                bytes = b;
                slot = cur.slot;
                par = cur.par;
                reuse = cur.reuse;
            }
            ++idx;
            cursor_next(cur, sh.NS);
        });
        c = cur;
        if (base >= idx) return true;
        if (!issue_batch(sh, src != nullptr, slot, par, reuse, src, bytes)) return false;
        if (base + sh.NS >= idx) return true;
    }
}

// Layer l's prefetch buffer (see CtaPlan) into sh.pb.
__device__ __forceinline__ void pb_issue(const KParams &kp, const Sh &sh, int l)
{
    const Geo &g = kp.g;
    const CtaPlan &b = *sh.cp;
    const LayerPtrs &Lp = kp.layer[l];
    mbar_expect_tx(sh.pb_full, (unsigned)b.bytes);
    bulk_load(sh.pb, Lp.gamma, (unsigned)(g.H * 2), sh.pb_full);
    if (b.nh > 0) {
        const size_t esz = g.qb ? 1 : 4;
        bulk_load(sh.pb + b.off_router, Lp.router_t + (size_t)b.h0 * g.Erp * esz, (unsigned)(b.nh * g.Erp * esz),
                  sh.pb_full);
        if (g.qb)
            bulk_load(sh.pb + b.off_rsb, Lp.router_t + g.rt_sb + (size_t)b.g0 * g.Erp * 4, (unsigned)(b.ng * g.Erp * 4),
                      sh.pb_full);
    }
    if (b.dpb > 0)
        bulk_load(sh.pb + b.off_sdown, Lp.sdown + (size_t)b.h0 * g.sd_bytes, (unsigned)(b.dpb * g.sd_bytes), sh.pb_full);
    if (b.upb > 0)
        bulk_load(sh.pb + b.off_units, Lp.sgu + (size_t)b.ua * 2 * g.sg_bytes, (unsigned)(b.upb * 2 * g.sg_bytes),
                  sh.pb_full);
}

// The producer warp (all 32 lanes, in step).  Lane 0 fills the prefetch
// buffer: layer 0's at once, layer l + 1's once layer l's stages are all
// issued and every compute warp is done with layer l's buffer.  Per layer
// the copies go out in the order the layer needs them: shared rows past the
// buffer, then (after routing) the routed gate/up stages, an L2 prefetch of
// every routed down stage (the ring holds only part of a layer), the shared
// down rows past the buffer, the routed down stages and the next layer's
// buffer.
__device__ __forceinline__ void producer(const KParams &kp, const Sh &sh, int lane)
{
    Cursor c = cursor0();
    int pb_issued = 1;
    if (lane == 0) pb_issue(kp, sh, 0);
    if (kp.mode == kModeLayers) {
#pragma unroll 1
        for (int l = 0; l < kp.L; ++l) {
            const LayerPtrs &Lp = kp.layer[l];
            if (!issue_pass(sh, c, lane, [&](auto &&f) { sched_p1x(kp, sh, Lp, f); })) break;
            if (lane == 0) stamp(kp, l, 9);
            // With one token row the routing always yields k distinct experts,
            // so each lane's gate/up stage (slot, units, ring position) is
            // known before the routing ends; after it only the expert id is
            // read and the copy goes out.
            int my_s = 0, my_j = 0, my_n = 0, nst = 0;
            if (kp.M == 1) p2_units(kp, sh, kp.g.k, [&](int s, int j, int n) {
                if (nst == lane) { my_s = s; my_j = j; my_n = n; }
                ++nst;
            });
            const bool fast = kp.M == 1 && nst <= sh.NS;
            Cursor mine = c;
#pragma unroll 1
            for (int i = 0; fast && i < lane; ++i) cursor_next(mine, sh.NS);
            if (!wait_bar(sh, sh.route, (unsigned)l & 1u, 2)) break;
            if (lane == 0) stamp(kp, l, 10);
            if (fast) {
                const int ub = 2 * kp.g.g_bytes;
                const uint8_t *src =
                    lane < nst ? Lp.gu + ((size_t)chk(sh, sh.slot_e[my_s], expert_blocks(kp, Lp), 7) * kp.g.I + my_j) * ub
                               : nullptr;
                if (!issue_batch(sh, lane < nst, mine.slot, mine.par, mine.reuse, src, my_n * ub)) break;
#pragma unroll 1
                for (int i = 0; i < nst; ++i) cursor_next(c, sh.NS);
            } else if (!issue_pass(sh, c, lane, [&](auto &&f) { sched_p2(kp, sh, Lp, f); })) {
                break;
            }
            if (lane == 0) stamp(kp, l, 14);
            int turn = 0;
            sched_p3(kp, sh, Lp, [&](const uint8_t *src, int bytes, int, int, int) {
                if (turn == lane) prefetch_l2(src, (unsigned)bytes);
                if (++turn == 32) turn = 0;
            });
            if (!issue_pass(sh, c, lane, [&](auto &&f) { sched_p1b(kp, sh, Lp, f); })) break;
            if (!issue_pass(sh, c, lane, [&](auto &&f) { sched_p3(kp, sh, Lp, f); })) break;
            if (lane == 0) stamp(kp, l, 11);
            if (l + 1 < kp.L) {
                if (!wait_bar(sh, sh.pb_empty, (unsigned)l & 1u, 3)) break;
                if (lane == 0 && !aborted(sh)) pb_issue(kp, sh, l + 1);
                pb_issued = l + 2;
            }
            if (aborted(sh)) break;
        }
    }
    // Let the copies still in flight land before the CTA can exit: slot s
    // was last filled in the cursor's round if s < c.slot, else in the round
    // before (if there was one).  Lane 0 waits for the last prefetch buffer.
    if (lane == 0) {
        const unsigned long long t0 = now_ns();
#pragma unroll 1
        while (!mbar_try_wait(sh.pb_full, (unsigned)(pb_issued - 1) & 1u))
            if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) break;
    }
#pragma unroll 1
    for (int s = lane; s < sh.NS; s += 32) {
        const bool cur = s < c.slot;
        if (!cur && !c.reuse) continue;
        const unsigned par = cur ? c.par : c.par ^ 1u;
        const unsigned long long t0 = now_ns();
#pragma unroll 1
        while (!mbar_try_wait(&sh.full[s], par))
            if (now_ns() - t0 > (unsigned long long)sh.timeout_ns) break;
    }
}

// -------------------------------------------------------- compute warps

// Trace bookkeeping of one phase's stages (diagnostic stamps of the first
// `tmax` stages a warp takes, at events tbase, tbase + 1, tbase + 2).
struct StageTrace {
    const KParams *kp;
    int l, count, base, max;
};

// Stage q belongs to warp q % NCW (NS is a multiple of NCW, so the warp
// itself consumed the previous round of the slot before it waits on this one).
template <typename F>
__device__ __forceinline__ void consume(const Sh &sh, Cursor &c, int where, F &&f, StageTrace *tr = nullptr)
{
    const bool mine = c.turn == (int)(threadIdx.x >> 5);
    const int slot = c.slot;
    const unsigned par = c.par;
    cursor_next(c, sh.NS);
    if (!mine) return;
    const bool st = tr && tr->kp && tr->count < tr->max;
    if (st) wstamp(*tr->kp, tr->l, tr->base);
    if (!aborted(sh) && wait_bar(sh, &sh.full[slot], par, where)) {
        if (st) wstamp(*tr->kp, tr->l, tr->base + 1);
        f(sh.ring + (size_t)slot * sh.S);
    }
    __syncwarp();
    if (st) { wstamp(*tr->kp, tr->l, tr->base + 2); ++tr->count; }
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[slot], 1);
}

// P0 and P1 (after router_partials).  With M at most half the compute
// warps, the first M warps each take one token row: they sum the CTA's
// router logits of that row from every CTA's partials, publish them and
// route (waiting on every CTA's logits), while the other warps build hn
// (the RMSNorm of the whole input, gathered from every CTA's outputs) and
// then compute the CTA's shared-expert gate/up units from the prefetch
// buffer, one range of units per warp, publishing their SwiGLU activations.
// With more rows every warp builds hn, the first M publish logits, every
// warp computes the shared units and the first M route after.  Shared units
// past the buffer come through the ring, one stage to each compute warp in
// turn.
__device__ void phase1(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, Cursor &q, const Ws &w, int l,
                       const void *xin, unsigned xtag)
{
    const Geo &g = kp.g;
    const uint32_t all = (1u << kp.M) - 1u;
    const int warp = threadIdx.x >> 5, M = kp.M;
    const CtaPlan &b = *sh.cp;
    const bool early = 2 * M <= NCW;
    const int w0 = early ? M : 0;   // first warp building hn
    const unsigned tag = layer_tag(sh, l);
    wstamp(kp, l, 14);
    if (early && warp < M) {
        reduce_logits(kp, sh, w.part, w.logits, warp, l);
        if (threadIdx.x == 0) stamp(kp, l, 22);
        route(kp, sh, w.logits, l);
    } else {
        build_hn(kp, sh, xin, xtag, reinterpret_cast<const uint16_t *>(sh.pb), w0);
        if (threadIdx.x == 32 * w0) stamp(kp, l, 1);
        if (!early && warp < M) reduce_logits(kp, sh, w.part, w.logits, warp, l);
        const int i0 = warp - w0, nw = NCW - w0;
        if (kp.mode == kModeLayers && b.upb > 0) {
            int u0, u1;
            split(b.upb, nw, i0, u0, u1);
            if (u1 > u0)
                gu_units(sh, g.H, g.sb, sh.pb + b.off_units + (size_t)u0 * 2 * g.sg_bytes, u1 - u0, g.sg_bytes, all,
                         w.act_s + b.ua + u0, g.Is, kp.ws_l.act_s_cs, tag);
        }
    }
    wstamp(kp, l, 15);
    // hn complete (the routing warps go on to shared units that came through
    // the ring, which read it)
    cbar();
    if (!early && warp < M) route(kp, sh, w.logits, l);
    if (kp.mode != kModeLayers) return;
    if (b.ub - b.ua > b.upb)
        sched_p1x(kp, sh, Lp, [&](const uint8_t *, int, int, int first, int n) {
            consume(sh, q, 10, [&](const uint8_t *st) {
                gu_units(sh, g.H, g.sb, st, n, g.sg_bytes, all, w.act_s + b.ua + first, g.Is, kp.ws_l.act_s_cs, tag);
            });
        });
}

// The shared expert's down rows held in the prefetch buffer, by the `nw`
// warps that finished their routed gate/up stages first (those with one
// stage fewer than the others; all warps when every warp has as many), this
// one as number `rank`: they stage the shared activations (published in P1)
// among themselves and split the rows.
__device__ void shared_down_light(const KParams &kp, const Sh &sh, const Ws &w, int l, int rank, int nw)
{
    const Geo &g = kp.g;
    const int M = kp.M, lane = threadIdx.x & 31;
    stage_acts(sh, M, g.Is, rank * 32 + lane, nw * 32, layer_tag(sh, l),
               [&](int p) -> const uint64_t * {
                   return w.act_s + (blockIdx.x % kActCopies) * kp.ws_l.act_s_cs + (size_t)p * g.Is;
               });
    asm volatile("bar.sync 4, %0;" ::"r"(nw * 32) : "memory");
    const uint32_t all = (1u << M) - 1u;
    const CtaPlan &b = *sh.cp;
    const int ch = (b.dpb + nw - 1) / nw, r0 = rank * ch;
    if (r0 < b.dpb)
        dn_rows(sh, g.sb, sh.pb + b.off_sdown + (size_t)r0 * g.sd_bytes, min(ch, b.dpb - r0), g.sd_bytes, g.Is, all, 0,
                sh.ysh + r0 * kMaxRows, kMaxRows, 1, 0u);
}

// Shared down rows held in the prefetch buffer, spread over compute warps
// w0 .. NCW-1 in equal chunks.
__device__ void shared_down_pb(const KParams &kp, const Sh &sh, int w0)
{
    const Geo &g = kp.g;
    const uint32_t all = (1u << kp.M) - 1u;
    const CtaPlan &b = *sh.cp;
    const int warp = threadIdx.x >> 5, nw = NCW - w0, ch = (b.dpb + nw - 1) / nw;
    const int r0 = (warp - w0) * ch;
    if (warp >= w0 && ch > 0 && r0 < b.dpb)
        dn_rows(sh, g.sb, sh.pb + b.off_sdown + (size_t)r0 * g.sd_bytes, min(ch, b.dpb - r0), g.sd_bytes, g.Is, all, 0,
                sh.ysh + r0 * kMaxRows, kMaxRows, 1, 0u);
}

__device__ void phase1b(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, Cursor &q, int l)
{
    const Geo &g = kp.g;
    const uint32_t all = (1u << kp.M) - 1u;
    StageTrace tr{kp.trace ? &kp : nullptr, l, 0, 11, 1};
    sched_p1b(kp, sh, Lp, [&](const uint8_t *, int, int, int first, int n) {
        consume(sh, q, 15, [&](const uint8_t *st) {
            dn_rows(sh, g.sb, st, n, g.sd_bytes, g.Is, all, 0, sh.ysh + first * kMaxRows, kMaxRows, 1, 0u);
        }, &tr);
    });
}

// P2.  Returns the number of stages and the turn of the first one.
__device__ void phase2(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, Cursor &q, const Ws &w, int l, int &n2,
                       int &turn0)
{
    const Geo &g = kp.g;
    const unsigned tag = layer_tag(sh, l);
    StageTrace tr{kp.trace ? &kp : nullptr, l, 0, 2, 1};
    n2 = 0;
    turn0 = q.turn;
    sched_p2(kp, sh, Lp, [&](const uint8_t *, int, int s, int first, int n) {
        ++n2;
        consume(sh, q, 20, [&](const uint8_t *st) {
            uint64_t *act = w.act + (size_t)s * kp.M * g.I;
            gu_units(sh, g.H, g.rb, st, n, g.g_bytes, sh.slot_mask[s], act + first, g.I, kp.ws_l.act_cs, tag);
        }, &tr);
    });
}

// P3: the routed down rows of this CTA's output slice.  The activations of
// the selected experts (tagged words from the CTAs that computed them, waited
// for) are staged in batches of whole slots, as many pairs as the staging
// buffer holds; then each slot's down stage gives yl[pair][h] for the
// slot's rows (pair = slot_rowbase[s] + rank of the row in the slot's mask).
__device__ bool phase3(const KParams &kp, const Sh &sh, const LayerPtrs &Lp, Cursor &q, const Ws &w, int l)
{
    const Geo &g = kp.g;
    const int U = sh.flags[1], hr = sh.hrows;
    const unsigned tag = layer_tag(sh, l);
    StageTrace tr{kp.trace ? &kp : nullptr, l, 0, 7, 1};
    int s0 = 0;
#pragma unroll 1
    while (s0 < U) {
        int s1 = s0;
        const int p0 = sh.slot_rowbase[s0];
        while (s1 < U && sh.slot_rowbase[s1 + 1] - p0 <= sh.act_pairs) ++s1;
        const int np = sh.slot_rowbase[s1] - p0;
        cbar();
        // staged pair p -> (slot, token row)
#pragma unroll 1
        for (int s = s0 + (int)threadIdx.x; s < s1; s += NCT) {
            uint32_t mk = sh.slot_mask[s];
#pragma unroll 1
            for (int p = sh.slot_rowbase[s] - p0; mk; mk &= mk - 1u, ++p)
                sh.pair_src[chk(sh, p, sh.act_pairs, 9)] = s * kMaxRows + __ffs(mk) - 1;
        }
        cbar();
        stage_acts(sh, np, g.I, threadIdx.x, NCT, tag, [&](int p) -> const uint64_t * {
            const int ps = sh.pair_src[p];
            return w.act + (blockIdx.x % kActCopies) * kp.ws_l.act_cs +
                   ((size_t)(ps / kMaxRows) * kp.M + ps % kMaxRows) * g.I;
        });
        if (cbar_or(aborted(sh))) return false;
        sched_p3(kp, sh, Lp, [&](const uint8_t *, int, int s, int first, int n) {
            if (s < s0 || s >= s1) return;
            consume(sh, q, 30, [&](const uint8_t *st) {
                dn_rows(sh, g.rb, st, n, g.d_bytes, g.I, sh.slot_mask[s], sh.slot_rowbase[s] - p0,
                        sh.yl + (size_t)sh.slot_rowbase[s] * hr + first, 1, hr, 0u);
            }, &tr);
        });
        s0 = s1;
    }
    cbar();
    return true;
}

// out = x + sum_j w_j y_j (expert-id order) + sigma y_shared for this CTA's
// outputs; thread t holds the row pair (2 pl, 2 pl + 1) of token row m,
// t = pl * M + m, with residuals xr.  Every y_j of these outputs was computed
// by this CTA (P3).  The bf16 pairs go out as tagged words (the next layer's
// input, or the input of the final RMSNorm) and, for the last layer, as
// plain bf16 to `plain`.
__device__ void combine(const KParams &kp, const Sh &sh, int l, const float (&xr)[2], uint64_t *tagged,
                        uint16_t *plain)
{
    const Geo &g = kp.g;
    const int M = kp.M, k = g.k, t = threadIdx.x, hr = sh.hrows;
    const int h0 = sh.cp->h0, np = sh.cp->nh / 2;
    const unsigned tag = layer_tag(sh, l);
    if (t >= np * M) return;
    const int pl = t / M, m = t % M;
    float acc[2] = {0.f, 0.f};
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        const float wv = sh.row_w[m * kMaxK + j];
        const float *y = sh.yl + (size_t)chk(sh, sh.row_pair[m * kMaxK + j], sh.slot_rowbase[sh.flags[1]], 10) * hr + 2 * pl;
        acc[0] = fmaf(wv, y[0], acc[0]);
        acc[1] = fmaf(wv, y[1], acc[1]);
    }
    uint32_t o[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int hl = 2 * pl + hh;
        float r = acc[hh];
        if (g.has_shared) r = fmaf(sh.sigma[m], sh.ysh[hl * kMaxRows + m], r);
        o[hh] = f2bf(xr[hh] + r);
    }
    const uint32_t pair = o[0] | (o[1] << 16);
    if (tagged) st_tag(tagged + (size_t)m * (g.H / 2) + h0 / 2 + pl, pair, tag);
    if (plain) *reinterpret_cast<uint32_t *>(plain + (size_t)m * g.H + h0 + 2 * pl) = pair;
    // the CTA's slice of the next layer's input, for its partial router dots
    // and residuals
    float *xv = sh.ru + kMaxRows * hr + m * hr + 2 * pl;
    xv[0] = bf2f((uint16_t)o[0]);
    xv[1] = bf2f((uint16_t)o[1]);
}

// out_n = bf16(out * rinv * gamma_next) for this CTA's outputs, with rinv from
// every CTA's bf16 outputs (tagged words of the last layer): the same
// computation as the next layer's RMSNorm (build_hn with gamma_next), of
// which this CTA keeps its own slice.
__device__ void final_normed(const KParams &kp, const Sh &sh, const uint64_t *xt, unsigned tag,
                             const uint16_t *gamma_next)
{
    const int H = kp.g.H, M = kp.M, G = H / kGroup;
    build_hn(kp, sh, xt, tag, gamma_next, 0);
    if (cbar_or(aborted(sh))) return;
    const int h0 = sh.cp->h0, nh = sh.cp->nh;
#pragma unroll 1
    for (int t = threadIdx.x; t < nh * M; t += NCT) {
        const int hl = t / M, m = t % M, h = h0 + hl;
        // hn_m[h] * 2^100 in the arranged layout: group h / 64, quad (h % 64) / 4
        const float4 v = sh.xs[(size_t)m * (H / 4) + ((h & 63) >> 2) * G + (h >> 6)];
        const float c = (h & 3) == 0 ? v.x : (h & 3) == 1 ? v.y : (h & 3) == 2 ? v.z : v.w;
        kp.out_normed[(size_t)m * H + h] = f2bf(c * 0x1p-100f);
    }
}

// No grid barrier between layers or phases: every piece of data one CTA
// publishes for others (router logits, shared and routed activations, the
// layer output) is a tagged word, and readers wait on the words themselves.
// (A word is rewritten only after every reader of its previous value is
// done: CTA A writes layer l + 1's copy only after its P0 of layer l + 1,
// which read every CTA's layer-l output, written after that CTA's last
// read of layer l.)  The fused final RMSNorm reads the last layer's output
// the same way.
__device__ __forceinline__ void compute(const KParams &kp, const Sh &sh)
{
    const Ws w = ws_views(kp);
    Cursor q = cursor0();
    const int np = sh.cp->nh / 2, M = kp.M;
    const int warp = threadIdx.x >> 5;
#pragma unroll 1
    for (int l = 0; l < kp.L; ++l) {
        const LayerPtrs &Lp = kp.layer[l];
        const bool last = l == kp.L - 1;
        const unsigned xtag = l == 0 ? 0u : layer_tag(sh, l - 1);
        const void *xin = l == 0 ? static_cast<const void *>(kp.x) : static_cast<const void *>(w.ping[(l - 1) & 1]);
        const bool t0 = threadIdx.x == 0;
        if (t0) stamp(kp, l, 0);
        // layer l's gamma, router slice and shared units
        const bool pb_ok = wait_bar(sh, sh.pb_full, (unsigned)l & 1u, 5);
        if (t0) stamp(kp, l, 18);
        if (cbar_or(!pb_ok)) return;
        router_partials(kp, sh, w.part, l);
        if (t0) stamp(kp, l, 19);
        phase1(kp, sh, Lp, q, w, l, xin, xtag);
        if (t0) stamp(kp, l, 2);
        if (t0) stamp(kp, l, 3);
        if (cbar_or(aborted(sh))) return;
        if (t0) stamp(kp, l, 4);
        if (kp.mode == kModeRouter) {
            if ((threadIdx.x & 31) == 0) mbar_arrive(sh.pb_empty, 1);
            break;
        }
        // residuals of this thread's output pair
        float xr[2] = {0.f, 0.f};
        if ((int)threadIdx.x < np * M) {
            // this CTA's slice of the layer input, kept in shared memory
            const int pl = threadIdx.x / M, m = threadIdx.x % M;
            const float *xv = sh.ru + kMaxRows * sh.hrows + m * sh.hrows + 2 * pl;
            xr[0] = xv[0];
            xr[1] = xv[1];
        }
        wstamp(kp, l, 0);
        wstamp(kp, l, 1);
        int n2 = 0, turn0 = 0;
        phase2(kp, sh, Lp, q, w, l, n2, turn0);
        wstamp(kp, l, 5);
        if (t0) stamp(kp, l, 5);
        // The shared expert's down rows, off the routed path: its activations
        // (waited for from every CTA) into the staging buffer, then the rows
        // held in the prefetch buffer and any that came through the ring.
        if (kp.g.has_shared && sh.cp->dpb == sh.cp->nh) {
            // the warps done with P2 first take the shared expert's down rows
            const int r0 = n2 % NCW, d = (warp - turn0 + NCW) % NCW;
            const int nw = r0 == 0 ? NCW : NCW - r0;
            if (r0 == 0 || d >= r0) shared_down_light(kp, sh, w, l, r0 == 0 ? d : d - r0, nw);
        } else if (kp.g.has_shared) {
            stage_acts(sh, M, kp.g.Is, threadIdx.x, NCT, layer_tag(sh, l),
                       [&](int p) -> const uint64_t * {
                           return w.act_s + (blockIdx.x % kActCopies) * kp.ws_l.act_s_cs + (size_t)p * kp.g.Is;
                       });
            cbar();
            shared_down_pb(kp, sh, 0);
            phase1b(kp, sh, Lp, q, l);
        }
        // every warp is done with the prefetch buffer of layer l, and with
        // the staging buffer (reused by P3)
        if ((threadIdx.x & 31) == 0) mbar_arrive(sh.pb_empty, 1);
        cbar();
        if (t0) stamp(kp, l, 6);
        wstamp(kp, l, 6);
        if (!phase3(kp, sh, Lp, q, w, l)) return;
        wstamp(kp, l, 10);
        if (cbar_or(aborted(sh))) return;
        const bool normed = last && kp.out_normed;
        combine(kp, sh, l, xr, last && !normed ? nullptr : w.ping[l & 1], last ? kp.out : nullptr);
        if (t0) stamp(kp, l, 7);
        if (normed) final_normed(kp, sh, w.ping[l & 1], layer_tag(sh, l), Lp.gamma_next);
        if (t0) stamp(kp, l, 8);
    }
}

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ KParams kp)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = carve(kp.g, kp.p);
    // The CTA's Sh lives in shared memory: every function reaches it through
    // a reference, with no copy in local memory.
    Sh &sh = *reinterpret_cast<Sh *>(smem + L.shs);
    if (threadIdx.x == 0) {
        CtaPlan *cplan = reinterpret_cast<CtaPlan *>(smem + L.cplan);
        cta_plan(kp, *cplan);
        sh.cp = cplan;
        uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar);
        sh.full = bars;
        sh.empty = bars + kp.p.NS;
        sh.route = bars + 2 * kp.p.NS;
        sh.pb_full = bars + 2 * kp.p.NS + 1;
        sh.pb_empty = bars + 2 * kp.p.NS + 2;
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
        sh.red = reinterpret_cast<float *>(smem + L.red);
        sh.ru = reinterpret_cast<float *>(smem + L.ru);
        sh.pair_src = reinterpret_cast<int *>(smem + L.pair_src);
        sh.xs = reinterpret_cast<float4 *>(smem + L.xs);
        sh.xsum = reinterpret_cast<float *>(smem + L.xsum);
        sh.act = reinterpret_cast<float4 *>(smem + L.act);
        sh.asum = reinterpret_cast<float *>(smem + L.asum);
        sh.ysh = reinterpret_cast<float *>(smem + L.ysh);
        sh.yl = reinterpret_cast<float *>(smem + L.yl);
        sh.pb = smem + L.pb;
        sh.ring = smem + L.ring;
        sh.NS = kp.p.NS;
        sh.S = kp.p.S;
        sh.hrows = kp.p.hrows;
        sh.act_pairs = kp.p.act_pairs;
        sh.timeout_ns = kp.timeout_ns;
        sh.ctrl = reinterpret_cast<Ctrl *>(kp.ws);
        sh.epoch = *reinterpret_cast<volatile unsigned *>(&sh.ctrl->seq) * 64u;
#pragma unroll 1
        for (int i = 0; i < kp.p.NS; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(sh.route, 1);
        mbar_init(sh.pb_full, 1);
        mbar_init(sh.pb_empty, NCW);
        sh.flags[0] = 0;
        sh.flags[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= NCT) {
        const int lane = threadIdx.x - NCT;
        producer(kp, sh, lane);
        return;
    }
    compute(kp, sh);
    if (threadIdx.x == 0) kernel_exit(kp, sh);
}

// ------------------------------------------------ fused Q/K/V projection
//
// y[m, r] = W[r] . x_m for the stacked rows of an attention's Q, K and V
// projections (or a Gated-DeltaNet input projection): "Qwen3.5-397B on M5
// Max" (openclawradar), 効果的な最適化: the Q/K/V projections fused so that
// the input row is read once.  x is the layer's normalised input (the MoE
// layer's fused out_n, bf16).  Each CTA streams its block of rows from HBM
// once, in up to kQkvChunks bulk copies with an mbarrier each; it stages the
// M input rows arranged and times 2^100 with their group sums, and its warps
// take the block's rows with the layer's row kernels, two token rows at a
// time (each code decoded once for both) or one; a row's arithmetic is the
// same in both, so its result does not depend on M.
constexpr int kQkvChunks = 4;
constexpr int kQkvThreads = 256;

struct QkvParams {
    const uint8_t *W;    // rows of row_bytes(K, bits)
    int rows, K, bits, rowb;
    const uint16_t *x;   // [M, K] bf16
    int M;
    float *y;            // [M, rows]
    int rows_per_cta;
    long long timeout_ns;
    int *err;            // set to 1 when a wait runs out (caller clears it)
};

__host__ __device__ inline size_t qkv_x_bytes(int M, int K) { return align_up((size_t)M * K * 4 + (size_t)M * (K / kGroup) * 4, 128); }

// ------------------------------------------------- grouped FMA products
//
// Grouped mode's expert products on the FMA pipes: slot u's expert over the
// token rows of its mask, the same dequantised dot products as the
// persistent kernel's row kernels (the one-vector plain1, or two token rows
// at a time with the codes decoded once for both: the same arithmetic per
// row).  One CTA per (block of rows, slot, group of up to 4 of the slot's
// token rows): its rows come in with one bulk copy (read once per group of
// token rows; a popular expert chosen by many rows gets several CTAs rather
// than one long one), then for each pair of token rows the input vectors
// are staged (arranged, times 2^100, group sums) and the warps split the
// rows.  Gate/up rows come in units (gate row, up row) and leave as
// silu(gate) * up.  With realistic routing a slot has one or two token rows,
// where the tensor-core products spend most of their work on padding.
struct FmaSet {
    const uint8_t *W;
    int rows, K, row_bytes, bits;
    const float *in;
    int in_u;
    const int32_t *experts;
    const uint32_t *masks;
    const int *U_dev;
    float *out;
};
struct FmaParams {
    FmaSet s[2];
    int nA, M, swiglu, block;   // block: units (gate/up) or rows per CTA
    long long timeout_ns;
    int *err;
};
constexpr int kFmaThreads = 256;

constexpr int kFmaRowGroup = 4;   // token rows of a slot per CTA (popular experts get several CTAs)

__host__ __device__ inline size_t fma_smem_bytes(int K, int block_bytes, int block_rows)
{
    return 128 + align_up((size_t)block_bytes, 128) + 2 * ((size_t)K * 4 + (size_t)(K / kGroup) * 4) +
           2 * (size_t)block_rows * 4;
}

__global__ void __launch_bounds__(kFmaThreads) grouped_fma_kernel(const __grid_constant__ FmaParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int y = blockIdx.y;
    const FmaSet &S = y < p.nA ? p.s[0] : p.s[1];
    const int u = y < p.nA ? y : y - p.nA;
    if (S.U_dev && u >= *S.U_dev) return;
    const int rpu = p.swiglu ? 2 : 1;                 // rows per unit
    const int units = S.rows / rpu;
    const int a0 = blockIdx.x * p.block;
    if (a0 >= units) return;
    const uint32_t mask = S.masks[u];
    // this CTA's token rows: set bits z * kFmaRowGroup .. + kFmaRowGroup - 1
    const int popc = __popc(mask), z = blockIdx.z;
    if (z * kFmaRowGroup >= popc) return;
    uint32_t mk = mask;
#pragma unroll 1
    for (int i = 0; i < z * kFmaRowGroup; ++i) mk &= mk - 1u;
    int left = min(kFmaRowGroup, popc - z * kFmaRowGroup);
    const int n = min(p.block, units - a0), nrows = n * rpu;
    const int e = S.experts[u];
    const int K = S.K, G = K / kGroup, tid = threadIdx.x, warp = tid >> 5;
    constexpr int NW = kFmaThreads / 32;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint8_t *rows = smem + 128;
    float4 *xs = reinterpret_cast<float4 *>(rows + align_up((size_t)p.block * rpu * S.row_bytes, 128));  // [2][K / 4]
    float *xsum = reinterpret_cast<float *>(xs + 2 * (K / 4));                                          // [2][G]
    float *tmp = xsum + 2 * G;                                                                          // [2][nrows]
    if (tid == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0) {
        const unsigned bytes = (unsigned)(nrows * S.row_bytes);
        mbar_expect_tx(bar, bytes);
        bulk_load(rows, S.W + ((size_t)e * S.rows + (size_t)a0 * rpu) * S.row_bytes, bytes, bar);
    }
    bool ok = true, landed = false;
    // warp w: block rows w, w + NW, ...
    const int cw = nrows > warp ? (nrows - warp + NW - 1) / NW : 0;
    const uint32_t rq = smem_u32(rows) + (uint32_t)(warp * S.row_bytes);
    const int rstride = NW * S.row_bytes;
#pragma unroll 1
    while (left > 0) {
        const int np = min(2, left);
        int ms[2];
        ms[0] = __ffs(mk) - 1;
        mk &= mk - 1u;
        ms[1] = ms[0];
        if (np == 2) {
            ms[1] = __ffs(mk) - 1;
            mk &= mk - 1u;
        }
        left -= np;
        if (ms[np - 1] >= p.M) break;
        // the np token rows' inputs: quads arranged (float4 t * G + g holds
        // inputs 64 g + 4 t ..), times 2^100; group sums over 16 quads
#pragma unroll 1
        for (int c = tid; c < np * (K / 4); c += kFmaThreads) {
            const int r = c / (K / 4), cc = c - r * (K / 4);
            const float4 v = __ldg(reinterpret_cast<const float4 *>(S.in + ((size_t)u * S.in_u + ms[r]) * K) + cc);
            float gs = (v.x + v.y) + (v.z + v.w);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) gs += __shfl_xor_sync(FULLMASK, gs, o);
            xs[r * (K / 4) + (cc & 15) * G + (cc >> 4)] =
                make_float4(v.x * kXScale, v.y * kXScale, v.z * kXScale, v.w * kXScale);
            if ((cc & 15) == 0) xsum[r * G + (cc >> 4)] = gs;
        }
        if (!landed) {
            // the rows' copy, waited for once (bounded)
            if (!mbar_try_wait(bar, 0u)) {
                const unsigned long long t0 = now_ns();
#pragma unroll 1
                while (!(ok = mbar_try_wait_sleep(bar, 0u, 2000)))
                    if (now_ns() - t0 > (unsigned long long)p.timeout_ns) break;
            }
            landed = true;
        }
        if (!__syncthreads_and(ok)) break;
        if (cw > 0) {
            // two token rows: the codes decoded once for both; one: the
            // one-vector kernel (the same arithmetic per row)
            if (np == 2) {
                const uint32_t xqa[2] = {smem_u32(xs), smem_u32(xs + K / 4)};
                const int soff[2] = {0, G};
                float xsg[2][kMaxGPL];
                lane_gsums<2>(smem_u32(xsum), soff, K, xsg);
                auto emit = [&](int rb, const float (&acc)[1][2]) {
                    tmp[rb * NW + warp] = acc[0][0];
                    tmp[nrows + rb * NW + warp] = acc[0][1];
                };
                const uint8_t *rp = rows + (size_t)warp * S.row_bytes;
                if (S.bits == 6) warp_rows<6, 1, 2>(rp, rstride, cw, K, xqa, xsg, emit);
                else if (S.bits == 8) warp_rows<8, 1, 2>(rp, rstride, cw, K, xqa, xsg, emit);
                else warp_rows<4, 1, 2>(rp, rstride, cw, K, xqa, xsg, emit);
            } else {
                if (S.bits == 6) plain1<6>(rq, cw, rstride, K, smem_u32(xs), smem_u32(xsum), tmp + warp, NW, 0u);
                else if (S.bits == 8) plain1<8>(rq, cw, rstride, K, smem_u32(xs), smem_u32(xsum), tmp + warp, NW, 0u);
                else plain1<4>(rq, cw, rstride, K, smem_u32(xs), smem_u32(xsum), tmp + warp, NW, 0u);
            }
        }
        __syncthreads();
#pragma unroll 1
        for (int r = 0; r < np; ++r) {
            float *o = S.out + ((size_t)u * p.M + ms[r]) * units + a0;
            const float *t = tmp + (size_t)r * nrows;
#pragma unroll 1
            for (int i = tid; i < n; i += kFmaThreads) {
                if (p.swiglu) {
                    const float gt = t[2 * i], up = t[2 * i + 1];
                    o[i] = gt / (1.0f + expf(-gt)) * up;
                } else {
                    o[i] = t[i];
                }
            }
        }
        __syncthreads();
    }
    if (!ok) {
        if (tid == 0) atomicOr(p.err, kStatusTimeout);
    }
    if (tid == 0 && (!ok || !landed)) {
        // the copy lands before the CTA exits
        const unsigned long long t0 = now_ns();
        while (!mbar_try_wait(bar, 0u) && now_ns() - t0 < (unsigned long long)p.timeout_ns) {}
    }
}

__global__ void __launch_bounds__(kQkvThreads) qkv_kernel(const __grid_constant__ QkvParams q)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int r0 = blockIdx.x * q.rows_per_cta;
    const int nr = min(q.rows_per_cta, q.rows - r0);
    if (nr <= 0) return;
    const int K = q.K, G = K / kGroup, M = q.M, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kQkvThreads / 32;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    float4 *xs = reinterpret_cast<float4 *>(smem + 128);
    float *xsum = reinterpret_cast<float *>(smem + 128 + (size_t)M * K * 4);
    uint8_t *rows = smem + 128 + qkv_x_bytes(M, K);
    const int cr = (nr + kQkvChunks - 1) / kQkvChunks;
    if (tid == 0) {
#pragma unroll 1
        for (int c = 0; c < kQkvChunks; ++c) mbar_init(&bars[c], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll 1
        for (int c = 0; c < kQkvChunks; ++c) {
            const int a = c * cr, n = min(cr, nr - a);
            if (n <= 0) break;
            mbar_expect_tx(&bars[c], (unsigned)(n * q.rowb));
            bulk_load(rows + (size_t)a * q.rowb, q.W + (size_t)(r0 + a) * q.rowb, (unsigned)(n * q.rowb), &bars[c]);
        }
    }
    // the input rows: 8 consecutive inputs per thread item, arranged (float4
    // t * G + g holds inputs 64 g + 4 t ..), times 2^100; group sums
    const int per_row = K / 8, total = M * per_row;
#pragma unroll 1
    for (int base = 0; base < total; base += kQkvThreads) {
        const int it = base + tid;
        float gs = 0.f;
        if (it < total) {
            const int m = it / per_row, c = it - m * per_row;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(q.x) + it);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = __uint_as_float(w[j] << 16);
                f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) gs += f[j];
            const int g = c >> 3, t = (c & 7) * 2;
            float4 *row = xs + (size_t)m * (K / 4);
            row[t * G + g] = make_float4(f[0] * kXScale, f[1] * kXScale, f[2] * kXScale, f[3] * kXScale);
            row[(t + 1) * G + g] = make_float4(f[4] * kXScale, f[5] * kXScale, f[6] * kXScale, f[7] * kXScale);
        }
        gs += __shfl_xor_sync(FULLMASK, gs, 4);
        gs += __shfl_xor_sync(FULLMASK, gs, 2);
        gs += __shfl_xor_sync(FULLMASK, gs, 1);
        if (it < total && (it & 7) == 0) {
            const int m = it / per_row, c = it - m * per_row;
            xsum[m * G + (c >> 3)] = gs;
        }
    }
    __syncthreads();
    const uint32_t xq0 = smem_u32(xs), xs0 = smem_u32(xsum);
    // every chunk (they travel together), bounded: a wait that runs out sets
    // the error word and the CTA leaves after its copies have landed
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < kQkvChunks && ok; ++c) {
        if (c * cr >= nr) break;
        if (mbar_try_wait(&bars[c], 0u)) continue;
        const unsigned long long t0 = now_ns();
#pragma unroll 1
        while (!(ok = mbar_try_wait_sleep(&bars[c], 0u, 2000)))
            if (now_ns() - t0 > (unsigned long long)q.timeout_ns) break;
    }
    if (!__syncthreads_and(ok)) {
        if (tid == 0) {
            atomicExch(q.err, 1);
#pragma unroll 1
            for (int c2 = 0; c2 < kQkvChunks && c2 * cr < nr; ++c2) {
                const unsigned long long t0 = now_ns();
                while (!mbar_try_wait(&bars[c2], 0u) && now_ns() - t0 < (unsigned long long)q.timeout_ns) {}
            }
        }
        return;
    }
    // warp w: rows w, w + NW, ... of the block; token rows two at a time
    // (the codes decoded once for both), the last one alone; each row's
    // arithmetic is the same in both kernels
    const int cnt = (nr - warp + NW - 1) / NW;
    if (cnt <= 0) return;
    const uint8_t *rp = rows + (size_t)warp * q.rowb;
    const uint32_t rbase = smem_u32(rp);
    float *yb = q.y + r0 + warp;
#pragma unroll 1
    for (int m = 0; m < M; m += 2) {
        if (m + 1 < M) {
            const uint32_t xqa[2] = {xq0 + (uint32_t)(m * K * 4), xq0 + (uint32_t)((m + 1) * K * 4)};
            const int soff[2] = {m * G, (m + 1) * G};
            float xsg[2][kMaxGPL];
            lane_gsums<2>(xs0, soff, K, xsg);
            auto emit = [&](int rb, const float (&acc)[1][2]) {
                yb[(size_t)m * q.rows + (size_t)rb * NW] = acc[0][0];
                yb[(size_t)(m + 1) * q.rows + (size_t)rb * NW] = acc[0][1];
            };
            if (q.bits == 8) warp_rows<8, 1, 2>(rp, NW * q.rowb, cnt, K, xqa, xsg, emit);
            else if (q.bits == 6) warp_rows<6, 1, 2>(rp, NW * q.rowb, cnt, K, xqa, xsg, emit);
            else warp_rows<4, 1, 2>(rp, NW * q.rowb, cnt, K, xqa, xsg, emit);
        } else {
            const uint32_t xq = xq0 + (uint32_t)(m * K * 4), xsq = xs0 + (uint32_t)(m * G * 4);
            float *dst = yb + (size_t)m * q.rows;
            if (K <= 32 * kGroup) {
                if (q.bits == 8) plain1<8>(rbase, cnt, NW * q.rowb, K, xq, xsq, dst, NW, 0u);
                else if (q.bits == 6) plain1<6>(rbase, cnt, NW * q.rowb, K, xq, xsq, dst, NW, 0u);
                else plain1<4>(rbase, cnt, NW * q.rowb, K, xq, xsq, dst, NW, 0u);
            } else {
                const uint32_t xqa[1] = {xq};
                const int soff[1] = {m * G};
                float xsg[1][kMaxGPL];
                lane_gsums<1>(xs0, soff, K, xsg);
                auto emit = [&](int rb, const float (&acc)[1][1]) { dst[(size_t)rb * NW] = acc[0][0]; };
                if (q.bits == 8) warp_rows<8, 1, 1>(rp, NW * q.rowb, cnt, K, xqa, xsg, emit);
                else if (q.bits == 6) warp_rows<6, 1, 1>(rp, NW * q.rowb, cnt, K, xqa, xsg, emit);
                else warp_rows<4, 1, 1>(rp, NW * q.rowb, cnt, K, xqa, xsg, emit);
            }
        }
    }
    (void)lane;
}

int g_num_sms[64];
bool g_attr_set[64];

}  // namespace

// Shared memory of a launch: small tables, hn rows, the activation staging
// buffer (act_pairs pairs), the prefetch buffer and the ring.  The ring gets
// up to ring_target first (enough bytes in flight to cover the HBM latency
// at one SM's share of the bandwidth), then the prefetch buffer up to one
// layer's P1 rows, then staging pairs up to every pair of a launch, then
// the ring takes whatever is left.
bool MOE_WBUILD(make_plan)(const Geo &g, int maxr, int num_sms, Plan &p)
{
    p.P = num_sms;
    p.maxr = maxr;
    p.ncw = NCW;
    p.max_slots = g.E < maxr * g.k ? g.E : maxr * g.k;
    p.hrows = 2 * ((g.H / 2 + num_sms - 1) / num_sms);   // whole row pairs per CTA
    int maxi = 2 * g.g_bytes;
    if (g.d_bytes > maxi) maxi = g.d_bytes;
    if (g.has_shared) {
        if (2 * g.sg_bytes > maxi) maxi = 2 * g.sg_bytes;   // one shared unit per stage at least
        if (g.sd_bytes > maxi) maxi = g.sd_bytes;
    }
    const int Im = imax_of(g);
    const int pair_bytes = Im * 4 + (Im / kGroup) * 4 + 4;
    if (num_sms > kMaxCtas || per_cta(g.Er + 1, num_sms) > kRouterRowsCta || p.hrows > kGroup) return false;
    const int pb_min = (int)align_up((size_t)g.H * 2, 16) + router_slice_bytes(p.hrows, 2, g.Erp, g.qb);
    // plus the CTA's shared down rows and shared gate/up units: with all of
    // them at hand, P1 needs no ring stages
    const int pb_all = pb_min + (g.has_shared ? p.hrows * g.sd_bytes + per_cta(g.Is, num_sms) * 2 * g.sg_bytes : 0);
    const int pairs_all = maxr * g.k + maxr;
    const int ring_target = 96 * 1024;
    // Every stage has one consumer warp: stage q goes to warp q % NCW, and a
    // warp waits on stage q only after it waited on stage q - NS of the same
    // slot (mbarrier parity tells apart only the current and previous phase),
    // so NS is a multiple of NCW.  A batch of the producer takes NS <= 32
    // stages, one per lane.
    static_assert(2 * NCW <= 32, "ring depth above the producer warp's width");
    p.NS = 2 * NCW;
    p.S = 0;
    p.pb_bytes = 0;
    p.act_pairs = 0;
    const int fixed = carve(g, p).total;
    int room = kSmemMax - 2048 - fixed - pb_min - maxr * pair_bytes;
    if (room < NCW * maxi) return false;
    // The staging buffer first: every activation pair of a launch, up to
    // kActCap bytes (each CTA's down rows need the activations of every
    // selected expert, and each batch of pairs costs a gather), keeping the
    // smallest ring; then the ring up to ring_target, then the prefetch
    // buffer, then the ring takes whatever is left.
    constexpr int kActCap = 80 * 1024;
    int more_pairs = pairs_all - maxr;
    const int cap_pairs = (kActCap - maxr * pair_bytes) / pair_bytes;
    if (more_pairs > cap_pairs) more_pairs = cap_pairs;
    if (more_pairs > (room - NCW * maxi) / pair_bytes) more_pairs = (room - NCW * maxi) / pair_bytes;
    if (more_pairs < 0) more_pairs = 0;
    p.act_pairs = maxr + more_pairs;
    room -= more_pairs * pair_bytes;
    const int ring_want = ring_target > NCW * maxi ? ring_target : NCW * maxi;
    int ring = room < ring_want ? room : ring_want;
    room -= ring;
    int pb_extra = pb_all - pb_min;
    if (pb_extra > room) pb_extra = room;
    p.pb_bytes = pb_min + pb_extra;
    room -= pb_extra;
    ring += room;
    // Stages large enough that a CTA's gate/up units at the most slots fit
    // one stage per compute warp (a warp with two stages would hold up the
    // CTA's P2 by a whole stage), if the ring allows it at any depth; else
    // stages of at least two gate/up units if it allows that.
    const int ub = 2 * g.g_bytes;
    const int units_cta = (int)(((long long)p.max_slots * g.I + num_sms - 1) / num_sms);
    const int want_all = ((units_cta + NCW - 1) / NCW) * ub;
    const int want = 2 * ub > maxi ? 2 * ub : maxi;
    int ns_pick = 0;
#pragma unroll 1
    for (int ns = 2 * NCW; ns >= NCW && !ns_pick; ns -= NCW)
        if (ring / ns >= want_all && ring / ns >= maxi) ns_pick = ns;
#pragma unroll 1
    for (int ns = 2 * NCW; ns >= NCW && !ns_pick; ns -= NCW)
        if (ring / ns >= want) ns_pick = ns;
#pragma unroll 1
    for (int ns = ns_pick ? ns_pick : 2 * NCW; ns >= NCW; ns -= NCW) {
        int S = ring / ns;
        S -= S % 16;
        if (S < maxi) continue;
        p.NS = ns;
        p.S = S;
        p.smem_bytes = carve(g, p).total;
        if (p.smem_bytes <= kSmemMax) return true;
    }
    return false;
}

int MOE_WBUILD(launch_decode)(const KParams &kp, cudaStream_t stream)
{
    if (kp.p.ncw != NCW) return MOE_ERR_INVALID_ARG;
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
    // the launch's tags come from the workspace's launch sequence (device side)
    e = cudaLaunchKernelEx(&cfg, moe_decode_kernel, kp);
    note_launch();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

#if MOE_NCW == 11
// (once in the library: the 8-warp build leaves these out)
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

int qkv_smem_bytes(int M, int K, int rows_per_cta, int rowb)
{
    return (int)(128 + qkv_x_bytes(M, K) + (size_t)rows_per_cta * rowb);
}

// Grouped mode's products on the FMA pipes (see grouped_fma_kernel): set a
// over its nA slots and set b (if given) over its nB, in one launch.  Sets
// with K above 2048 (the one-vector kernel's limit) are refused
// (MOE_ERR_UNSUPPORTED): the caller uses the tensor-core products there.
int launch_grouped_fma(bool swiglu, int bits_a, const TcSetHost &a, int nA, int bits_b, const TcSetHost *b, int nB,
                       int M, int *err, long long timeout_ns, cudaStream_t stream)
{
    const TcSetHost *sets[2] = {&a, b};
    const int bits[2] = {bits_a, bits_b};
    FmaParams P;
    memset(&P, 0, sizeof P);
    int Kmax = 0, rowb_max = 0;
    for (int i = 0; i < 2; ++i) {
        if (!sets[i]) continue;
        const TcSetHost &t = *sets[i];
        // (K a multiple of 128: the staging's shuffles run on whole warps)
        if (t.K > 32 * kGroup || t.K % 128 || !(bits[i] == 4 || bits[i] == 6 || bits[i] == 8))
            return MOE_ERR_UNSUPPORTED;
        P.s[i] = FmaSet{t.W, t.rows, t.K, t.row_bytes, bits[i], t.in, t.in_u, t.experts, t.masks, t.U_dev, t.out};
        Kmax = max(Kmax, t.K);
        rowb_max = max(rowb_max, t.row_bytes);
    }
    const int rpu = swiglu ? 2 : 1;
    // rows per CTA: about 80 KB of them (two CTAs per SM), whole units
    int block = max(1, (80 * 1024) / (rpu * rowb_max));
    if (block > 1024 / rpu) block = 1024 / rpu;
    P.nA = nA;
    P.M = M;
    P.swiglu = swiglu ? 1 : 0;
    P.block = block;
    P.timeout_ns = timeout_ns;
    P.err = err;
    const size_t smem = fma_smem_bytes(Kmax, block * rpu * rowb_max, block * rpu);
    static std::once_flag attr_once[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    std::call_once(attr_once[dev], [&] {
        e = cudaFuncSetAttribute(grouped_fma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    });
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    int units_max = 0;
    for (int i = 0; i < 2; ++i)
        if (sets[i]) units_max = max(units_max, sets[i]->rows / rpu);
    const dim3 grid((unsigned)((units_max + block - 1) / block), (unsigned)(nA + (b ? nB : 0)),
                    (unsigned)((M + kFmaRowGroup - 1) / kFmaRowGroup));
    grouped_fma_kernel<<<grid, kFmaThreads, smem, stream>>>(P);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

int launch_qkv(const uint8_t *W, int rows, int K, int bits, const uint16_t *x, int M, float *y, int *err,
               long long timeout_ns, cudaStream_t stream)
{
    const int sms = device_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    const int rowb = row_bytes(K, bits);
    // rows per CTA: an even share over the SMs, fewer if they do not fit in
    // shared memory beside the staged input rows
    int per = (rows + sms - 1) / sms;
    const int room = kSmemMax - 128 - (int)qkv_x_bytes(M, K);
    if (room < rowb) return MOE_ERR_UNSUPPORTED;
    if (per * rowb > room) per = room / rowb;
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(qkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
        attr_set[dev] = true;
    }
    QkvParams q{W, rows, K, bits, rowb, x, M, y, per, timeout_ns, err};
    const int grid = (rows + per - 1) / per;
    qkv_kernel<<<grid, kQkvThreads, qkv_smem_bytes(M, K, per, rowb), stream>>>(q);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

#endif  // MOE_NCW == 11

}  // namespace moe

