// Host side of the C ABI declared in include/moe.h: argument checks,
// blob/workspace layouts, row chunking and kernel launches.  No device
// memory is allocated here.
#include <atomic>
#include <cstdio>
#include <mutex>
#include <cstdlib>
#include <cstring>

#include "moe_internal.h"
#include "moe_unpack.cuh"

namespace moe {

namespace {
thread_local int t_last_cuda_error = 0;
thread_local long long t_launches = 0;
int g_skip_row = -1;
int g_inject_e = -1;   // checked build only (moe_debug_inject)
unsigned long long *g_trace = nullptr;
long long g_timeout_ns = 2000000000LL;
// Grouped mode for M above one launch's rows and at least this (0 = off).
// On the 35B shape the 40-layer stack runs 16 rows grouped in 240 us per
// layer against 259 in two 8-row launches, and 32 rows in 265 against 470.
int g_grouped_min_rows = 1;
std::atomic<int> g_grouped_tc{0};   // grouped mode's products: 0 FMA, 1 tensor cores

// Contraction widths 64 * 2^j up to 64 * 32 * kMaxGPL: a row splits into
// whole groups over 1, 2, 4, ..., 32 lanes.
bool width_ok(int K)
{
    for (int w = kGroup; w <= kGroup * 32 * kMaxGPL; w *= 2)
        if (K == w) return true;
    return false;
}

bool bits_ok(int b) { return b == 4 || b == 6 || b == 8; }

int check_status_word(void *ws)
{
    int st = 0;
    cudaError_t e = cudaMemcpy(&st, reinterpret_cast<uint8_t *>(ws) + offsetof(Ctrl, status), sizeof st,
                               cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    if (st & kStatusTimeout) return MOE_ERR_TIMEOUT;
    if (st & kStatusNotResident) return MOE_ERR_NOT_RESIDENT;
    if (st) return MOE_ERR_DEVICE;
    return MOE_OK;
}
}  // namespace

void note_cuda_error(int err) { t_last_cuda_error = err; }
bool grouped_products_tc() { return g_grouped_tc.load(std::memory_order_relaxed) != 0; }
void note_launch() { ++t_launches; }

int rows_per_launch(int H)
{
    int r = 16384 / H;
    if (r > kMaxRows) r = kMaxRows;
    return r < 1 ? 1 : r;
}

bool make_geo(const moe_layer_desc &d, Geo &g)
{
    if (d.H < 256 || !width_ok(d.H) || !width_ok(d.I) || d.I > d.H || d.I > 1024) return false;
    if (d.E < 1 || d.E > kMaxE || d.k < 1 || d.k > d.E || d.k > kMaxK) return false;
    if (!bits_ok(d.routed_bits)) return false;
    if (!(d.router_bits == 0 || bits_ok(d.router_bits))) return false;
    if (d.has_shared != 0 && d.has_shared != 1) return false;
    if (d.has_shared && (!bits_ok(d.shared_bits) || !width_ok(d.I_shared) || d.I_shared > d.H || d.I_shared > 1024))
        return false;
    if (!(d.eps > 0.0f)) return false;
    memset(&g, 0, sizeof g);
    g.H = d.H; g.I = d.I; g.E = d.E; g.k = d.k;
    g.has_shared = d.has_shared;
    g.Is = d.has_shared ? d.I_shared : 0;
    g.rb = d.routed_bits;
    g.sb = d.has_shared ? d.shared_bits : 8;
    g.qb = d.router_bits;
    g.Er = d.E + d.has_shared;
    g.Erp = (int)align_up((size_t)g.Er, 16);
    g.eps = d.eps;
    g.rr_bytes = row_bytes(g.H, g.qb);
    g.g_bytes = row_bytes(g.H, g.rb);
    g.d_bytes = row_bytes(g.I, g.rb);
    g.sg_bytes = d.has_shared ? row_bytes(g.H, g.sb) : 0;
    g.sd_bytes = d.has_shared ? row_bytes(g.Is, g.sb) : 0;
    size_t o = 0;
    auto put = [&](size_t bytes) { o = align_up(o, 256); size_t r = o; o += bytes; return r; };
    g.off_router = put((size_t)g.Er * g.rr_bytes);
    g.off_gamma = put((size_t)g.H * 2);
    g.off_gamma_next = put((size_t)g.H * 2);
    g.off_router_t = put(router_t_bytes(g.H, g.Erp, g.qb));
    g.rt_sb = (size_t)g.H * g.Erp;
    g.off_gu = put((size_t)g.E * g.I * 2 * g.g_bytes);
    g.off_down = put((size_t)g.E * g.H * g.d_bytes);
    g.off_sgu = put(d.has_shared ? (size_t)g.Is * 2 * g.sg_bytes : 0);
    g.off_sdown = put(d.has_shared ? (size_t)g.H * g.sd_bytes : 0);
    g.total = align_up(o, 256);
    return true;
}

void make_ws_layout(const Geo &g, int max_M, WsLayout &w)
{
    const int R = rows_per_launch(g.H);
    w.maxr = R;
    w.max_slots = g.E < R * g.k ? g.E : R * g.k;
    w.max_M = max_M;
    size_t o = kCtrlBytes;
    auto put = [&](size_t bytes) { o = align_up(o, 256); size_t r = o; o += bytes; return r; };
    // buffers CTAs exchange hold tagged 8-byte words (value | tag << 32)
    // router logits before the RMSNorm scale, and (last) the row's sum of
    // squares: [kLogitCopies][R][Er + 1]
    w.off_logits = put((size_t)kLogitCopies * R * (g.Er + 1) * 8);
    // activations: [kActCopies][slot][row][I] and [kActCopies][row][Is],
    // rows of one launch (at most min(max_M, R))
    const int Mr = max_M < R ? max_M : R;
    w.act_cs = (size_t)(g.E < Mr * g.k ? g.E : Mr * g.k) * Mr * g.I;
    w.act_s_cs = (size_t)Mr * (g.Is ? g.Is : 1);
    w.off_act = put((size_t)kActCopies * w.act_cs * 8);
    w.off_act_s = put((size_t)kActCopies * w.act_s_cs * 8);
    w.off_ping = put((size_t)2 * R * (g.H / 2) * 8);
    // partial router dots and sums of squares: [row][Er + 1][CTA], for the
    // rows of one launch
    w.off_part = put((size_t)kMaxCtas * (max_M < R ? max_M : R) * (g.Er + 1) * 8);
    w.off_stage_in = put((size_t)max_M * g.H * 2);
    w.off_stage_out = put((size_t)max_M * g.H * 2);
    w.grp_rows = w.grp_slots = 0;
    w.off_g_hn = w.off_g_sigma = w.off_g_idx = w.off_g_w = w.off_g_slotof = w.off_g_experts = w.off_g_masks = 0;
    w.off_g_count = w.off_g_act = w.off_g_act_s = w.off_g_y = w.off_g_ysh = w.off_g_ping = 0;
    if (max_M > R) {
        const int GR = max_M < kGroupRows ? max_M : kGroupRows;
        const int GS = g.E < GR * g.k ? g.E : GR * g.k;
        w.grp_rows = GR;
        w.grp_slots = GS;
        w.off_g_hn = put((size_t)GR * g.H * 4);
        w.off_g_sigma = put((size_t)GR * 4);
        w.off_g_idx = put((size_t)GR * g.k * 4);
        w.off_g_w = put((size_t)GR * g.k * 4);
        w.off_g_slotof = put((size_t)GR * g.k * 4);
        w.off_g_experts = put((size_t)(GS + 1) * 4);   // + the shared expert's entry
        w.off_g_masks = put((size_t)(GS + 1) * 4);
        w.off_g_count = put(4);
        w.off_g_act = put((size_t)GS * GR * g.I * 4);
        w.off_g_act_s = put((size_t)GR * (g.Is ? g.Is : 1) * 4);
        w.off_g_y = put((size_t)GS * GR * g.H * 4);
        w.off_g_ysh = put((size_t)GR * g.H * 4);
        w.off_g_ping = put((size_t)2 * GR * g.H * 2);
    }
    w.total = align_up(o, 256);
}

namespace {

// The layout without the grouped-mode regions (they sit at the end): what a
// call that stays on the persistent kernel needs.
void make_ws_layout_fma(const Geo &g, int max_M, WsLayout &w)
{
    make_ws_layout(g, max_M, w);
    if (w.grp_rows) {
        w.total = align_up(w.off_stage_out + (size_t)max_M * g.H * 2, 256);
        w.grp_rows = w.grp_slots = 0;
    }
}

bool use_grouped(int M, int R) { return M > R && g_grouped_min_rows > 0 && M >= g_grouped_min_rows; }

int prepare(const moe_layer *layer, int M, void *ws, size_t ws_bytes, KParams &kp, int &R)
{
    if (!layer || !ws || M < 1) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_ERR_INVALID_ARG;
    memset(&kp, 0, sizeof kp);
    kp.g = layer->geo;
    // the persistent kernel's regions; grouped mode checks its own (larger)
    // layout when it runs
    make_ws_layout_fma(kp.g, M, kp.ws_l);
    if (ws_bytes < kp.ws_l.total) return MOE_ERR_BUFFER_TOO_SMALL;
    R = kp.ws_l.maxr;
    kp.ws = reinterpret_cast<uint8_t *>(ws);
    kp.timeout_ns = g_timeout_ns;
    kp.skip_row = g_skip_row;
    kp.inject_e = g_inject_e;
    kp.trace = g_trace;
    return MOE_OK;
}

int plan_for(KParams &kp, int mc)
{
    const int sms = device_sms();
    if (sms <= 0) return MOE_ERR_CUDA;
    if (!decode_plan(kp.g, mc, sms, kp.p)) return MOE_ERR_UNSUPPORTED;
    kp.M = mc;
    return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Launch plans of the three test shapes (and of the 35B geometry at every
// routed width) for every row count of a launch and several SM counts,
// checked against what the kernel relies on: the ring depth a multiple of
// the compute warps and within one producer batch, stages that hold any
// single bulk copy, the shared-memory limit, a staging buffer that holds
// every row of a slot, a prefetch buffer that holds gamma and the CTA's
// slice of the input-major router, at most kRouterRowsCta router rows and at
// most one group of output rows per CTA, whole output row pairs per CTA, and
// 32-bit products in the work split.  Returns the number of violations.
int plan_selftest_host()
{
    const moe_layer_desc shapes[] = {
        {256, 128, 16, 2, 4, 8, 0, 0, 0, 1e-6f},
        {2048, 512, 256, 8, 6, 8, 8, 1, 512, 1e-6f},
        {2048, 512, 256, 8, 4, 8, 8, 1, 512, 1e-6f},
        {2048, 512, 256, 8, 8, 8, 8, 1, 512, 1e-6f},
        {4096, 1024, 512, 10, 4, 8, 8, 1, 1024, 1e-6f},
    };
    const int sm_counts[] = {132, 148, 152, 160};
    int bad = 0;
    for (const moe_layer_desc &d : shapes) {
        Geo g;
        if (!make_geo(d, g)) { ++bad; continue; }
        const int R = rows_per_launch(g.H);
        int maxi = 2 * g.g_bytes;
        if (g.d_bytes > maxi) maxi = g.d_bytes;
        if (2 * g.sg_bytes > maxi) maxi = 2 * g.sg_bytes;
        if (g.sd_bytes > maxi) maxi = g.sd_bytes;
        for (int sms : sm_counts)
            for (int mc = 1; mc <= R; ++mc) {
                Plan p;
                if (!decode_plan(g, mc, sms, p)) { ++bad; continue; }
                if (p.ncw != decode_warps(g, mc) || p.NS % p.ncw != 0 || p.NS > 32 || p.NS > kMaxStages) ++bad;
                if (p.S % 16 != 0 || p.S < maxi) ++bad;
                if (p.smem_bytes > kSmemMax) ++bad;
                if (p.act_pairs < p.maxr) ++bad;
                const int rows_cta = (g.Er + 1 + sms - 1) / sms;
                if (rows_cta > kRouterRowsCta || sms > kMaxCtas || p.hrows > kGroup) ++bad;
                if (p.pb_bytes < (int)align_up((size_t)g.H * 2, 16) + router_slice_bytes(p.hrows, 2, g.Erp, g.qb)) ++bad;
                if (p.hrows % 2 != 0 || (long long)p.hrows * sms < g.H) ++bad;
                const long long lim = 1ll << 32;
                const long long ns[] = {g.Er, g.Is, (long long)p.max_slots * g.I, g.H / 2};
                for (long long n : ns)
                    if (n * sms >= lim) ++bad;
            }
    }
    return bad;
}

// Host-side check of the workspace layouts over shapes and row counts: every
// region 256-byte aligned, in order, large enough for what its users write
// into it, and inside the total; the grouped regions sized for min(M, 32)
// rows and min(E, rows k) experts, and absent from the persistent-only
// layout.  Returns the number of violations.
int ws_layout_selftest_host()
{
    const moe_layer_desc shapes[] = {
        {256, 128, 16, 2, 4, 8, 0, 0, 0, 1e-6f},
        {2048, 512, 256, 8, 6, 8, 8, 1, 512, 1e-6f},
        {4096, 1024, 512, 10, 4, 8, 8, 1, 1024, 1e-6f},
    };
    const int rows[] = {1, 2, 4, 7, 8, 9, 16, 17, 31, 32, 33, 64, 100};
    int bad = 0;
    for (const moe_layer_desc &d : shapes) {
        Geo g;
        if (!make_geo(d, g)) { ++bad; continue; }
        const size_t Is = g.Is ? (size_t)g.Is : 1;
        for (int M : rows) {
            WsLayout w, f;
            make_ws_layout(g, M, w);
            make_ws_layout_fma(g, M, f);
            const int R = w.maxr;
            // the persistent kernel's regions, in order, each holding its data
            const size_t need[][2] = {
                {w.off_logits, (size_t)kLogitCopies * R * (g.Er + 1) * 8},
                {w.off_act, (size_t)kActCopies * (g.E < (M < R ? M : R) * g.k ? g.E : (M < R ? M : R) * g.k) *
                                (M < R ? M : R) * g.I * 8},
                {w.off_act_s, (size_t)kActCopies * (M < R ? M : R) * Is * 8},
                {w.off_ping, (size_t)2 * R * (g.H / 2) * 8},
                {w.off_part, (size_t)kMaxCtas * (M < R ? M : R) * (g.Er + 1) * 8},
                {w.off_stage_in, (size_t)M * g.H * 2},
                {w.off_stage_out, (size_t)M * g.H * 2},
            };
            size_t end = kCtrlBytes;
            for (const auto &r : need) {
                if (r[0] % 256 != 0 || r[0] < end) ++bad;
                end = r[0] + r[1];
            }
            if (f.total < end || f.total > w.total || f.total % 256 != 0 || f.grp_rows != 0) ++bad;
            if (w.max_slots != (g.E < R * g.k ? g.E : R * g.k)) ++bad;
            if (M <= R) {
                if (w.grp_rows != 0 || w.grp_slots != 0 || w.total != f.total) ++bad;
                continue;
            }
            const int GR = M < kGroupRows ? M : kGroupRows;
            const int GS = g.E < GR * g.k ? g.E : GR * g.k;
            if (w.grp_rows != GR || w.grp_slots != GS) ++bad;
            const size_t gneed[][2] = {
                {w.off_g_hn, (size_t)GR * g.H * 4},
                {w.off_g_sigma, (size_t)GR * 4},
                {w.off_g_idx, (size_t)GR * g.k * 4},
                {w.off_g_w, (size_t)GR * g.k * 4},
                {w.off_g_slotof, (size_t)GR * g.k * 4},
                {w.off_g_experts, (size_t)(GS + 1) * 4},
                {w.off_g_masks, (size_t)(GS + 1) * 4},
                {w.off_g_count, 4},
                {w.off_g_act, (size_t)GS * GR * g.I * 4},
                {w.off_g_act_s, (size_t)GR * Is * 4},
                {w.off_g_y, (size_t)GS * GR * g.H * 4},
                {w.off_g_ysh, (size_t)GR * g.H * 4},
                {w.off_g_ping, (size_t)2 * GR * g.H * 2},
            };
            for (const auto &r : gneed) {
                if (r[0] % 256 != 0 || r[0] < end) ++bad;
                end = r[0] + r[1];
            }
            if (w.total < end || w.total % 256 != 0) ++bad;
        }
    }
    return bad;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_pack_size(const moe_layer_desc *desc, size_t *weight_bytes)
{
    if (!desc || !weight_bytes) return MOE_ERR_INVALID_ARG;
    Geo g;
    if (!make_geo(*desc, g)) return MOE_ERR_UNSUPPORTED;
    *weight_bytes = g.total;
    return MOE_OK;
}

int moe_pack_weights(const moe_layer_desc *desc, const moe_src_layer *src, void *dst_dev, size_t dst_bytes,
                     moe_layer **out, moe_stream_t stream)
{
    if (!desc || !src || !dst_dev || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    Geo g;
    if (!make_geo(*desc, g)) return MOE_ERR_UNSUPPORTED;
    if (dst_bytes < g.total) return MOE_ERR_BUFFER_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(dst_dev) & 255) != 0) return MOE_ERR_INVALID_ARG;
    if (!src->gamma_dev) return MOE_ERR_INVALID_ARG;
    moe_layer *L = static_cast<moe_layer *>(calloc(1, sizeof(moe_layer)));
    if (!L) return MOE_ERR_INVALID_ARG;
    L->desc = *desc;
    L->geo = g;
    L->base = static_cast<uint8_t *>(dst_dev);
    L->bytes = dst_bytes;
    L->ptrs.router = L->base + g.off_router;
    L->ptrs.router_t = L->base + g.off_router_t;
    L->ptrs.gu = L->base + g.off_gu;
    L->ptrs.down = L->base + g.off_down;
    L->ptrs.sgu = g.has_shared ? L->base + g.off_sgu : nullptr;
    L->ptrs.sdown = g.has_shared ? L->base + g.off_sdown : nullptr;
    L->ptrs.gamma = reinterpret_cast<const uint16_t *>(L->base + g.off_gamma);
    L->ptrs.gamma_next = src->gamma_next_dev ? reinterpret_cast<const uint16_t *>(L->base + g.off_gamma_next) : nullptr;
    const int rc = launch_pack(*L, *src, reinterpret_cast<cudaStream_t>(stream));
    if (rc != MOE_OK) {
        free(L);
        return rc;
    }
    *out = L;
    return MOE_OK;
}

void moe_layer_destroy(moe_layer *layer) { free(layer); }

int moe_export_canonical(const moe_layer *layer, int tensor_id, int expert, uint8_t *codes_dev,
                         uint16_t *scales_dev, uint16_t *biases_dev, moe_stream_t stream)
{
    if (!layer || !codes_dev || !scales_dev || !biases_dev) return MOE_ERR_INVALID_ARG;
    return launch_export(*layer, tensor_id, expert, codes_dev, scales_dev, biases_dev,
                         reinterpret_cast<cudaStream_t>(stream));
}

int moe_workspace_size(const moe_layer_desc *desc, int max_M, size_t *ws_bytes)
{
    if (!desc || !ws_bytes || max_M < 1) return MOE_ERR_INVALID_ARG;
    Geo g;
    if (!make_geo(*desc, g)) return MOE_ERR_UNSUPPORTED;
    WsLayout w;
    make_ws_layout(g, max_M, w);
    *ws_bytes = w.total;
    return MOE_OK;
}

int moe_workspace_init(void *ws_dev, size_t ws_bytes, moe_stream_t stream)
{
    if (!ws_dev || ws_bytes < (size_t)kCtrlBytes) return MOE_ERR_INVALID_ARG;
    // the whole workspace: the control block (launch sequence, status) and
    // every exchanged word (tag 0 is never a launch's tag)
    cudaError_t e = cudaMemsetAsync(ws_dev, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

int moe_router_topk(const moe_layer *layer, const uint16_t *x_dev, int M, int32_t *idx_dev, float *w_dev,
                    void *ws_dev, size_t ws_bytes, moe_stream_t stream)
{
    if (!x_dev || !idx_dev || !w_dev || !aligned16(x_dev)) return MOE_ERR_INVALID_ARG;
    KParams kp;
    int R;
    int rc = prepare(layer, M, ws_dev, ws_bytes, kp, R);
    if (rc) return rc;
    kp.mode = kModeRouter;
    kp.L = 1;
    kp.layer[0] = layer->ptrs;
    const int H = kp.g.H, k = kp.g.k;
    for (int c0 = 0; c0 < M; c0 += R) {
        const int mc = M - c0 < R ? M - c0 : R;
        if ((rc = plan_for(kp, mc))) return rc;
        kp.x = x_dev + (size_t)c0 * H;
        kp.idx_out = idx_dev + (size_t)c0 * k;
        kp.w_out = w_dev + (size_t)c0 * k;
        if ((rc = decode_launch(kp, reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    return MOE_OK;
}

namespace {

int decode_layer_impl(const moe_layer *layer, const uint16_t *x_dev, int M, uint16_t *out_dev,
                      uint16_t *out_normed_dev, void *ws_dev, size_t ws_bytes, moe_stream_t stream, bool allow_grouped,
                      bool clear_status = false)
{
    if (!x_dev || !out_dev || !aligned16(x_dev) || !aligned16(out_dev)) return MOE_ERR_INVALID_ARG;
    if (out_normed_dev && (!layer || !layer->ptrs.gamma_next)) return MOE_ERR_INVALID_ARG;
    KParams kp;
    int R;
    int rc = prepare(layer, M, ws_dev, ws_bytes, kp, R);
    if (rc) return rc;
    // grouped mode (moe_set_grouped); never for a streamed layer, whose
    // experts are reached through its cache's slot map
    if (allow_grouped && !layer->ptrs.slot_of && use_grouped(M, R))
        return grouped_forward(&layer, 1, x_dev, M, out_dev, out_normed_dev, ws_dev, ws_bytes, g_timeout_ns,
                               reinterpret_cast<cudaStream_t>(stream));
    kp.mode = kModeLayers;
    kp.L = 1;
    kp.layer[0] = layer->ptrs;
    const int H = kp.g.H;
    // every launch plan is made before anything is enqueued, so a call that
    // fails its checks leaves the stream untouched
    const int tail = M % R;
    {
        KParams probe = kp;
        if ((rc = plan_for(probe, M < R ? M : R))) return rc;
        if (tail && M > R && (rc = plan_for(probe, tail))) return rc;
    }
    if (clear_status) {
        cudaError_t e = cudaMemsetAsync(static_cast<uint8_t *>(ws_dev) + offsetof(Ctrl, status), 0, 2 * sizeof(int),
                                        reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    }
    for (int c0 = 0; c0 < M; c0 += R) {
        const int mc = M - c0 < R ? M - c0 : R;
        if ((rc = plan_for(kp, mc))) return rc;
        kp.x = x_dev + (size_t)c0 * H;
        kp.out = out_dev + (size_t)c0 * H;
        kp.out_normed = out_normed_dev ? out_normed_dev + (size_t)c0 * H : nullptr;
        if ((rc = decode_launch(kp, reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    return MOE_OK;
}

}  // namespace

int moe_decode_layer(const moe_layer *layer, const uint16_t *x_dev, int M, uint16_t *out_dev,
                     uint16_t *out_normed_dev, void *ws_dev, size_t ws_bytes, moe_stream_t stream)
{
    return decode_layer_impl(layer, x_dev, M, out_dev, out_normed_dev, ws_dev, ws_bytes, stream, true);
}

int moe_stack_create(moe_layer *const *layers, int L, moe_stack **out)
{
    if (!layers || L < 1 || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    for (int l = 0; l < L; ++l) {
        if (!layers[l]) return MOE_ERR_INVALID_ARG;
        if (memcmp(&layers[l]->desc, &layers[0]->desc, sizeof(moe_layer_desc)) != 0) return MOE_ERR_INVALID_ARG;
    }
    moe_stack *s = static_cast<moe_stack *>(calloc(1, sizeof(moe_stack)));
    if (!s) return MOE_ERR_INVALID_ARG;
    s->layers = static_cast<moe_layer **>(calloc((size_t)L, sizeof(moe_layer *)));
    if (!s->layers) { free(s); return MOE_ERR_INVALID_ARG; }
    memcpy(s->layers, layers, sizeof(moe_layer *) * (size_t)L);
    s->L = L;
    *out = s;
    return MOE_OK;
}

int moe_stack_forward(moe_stack *stack, const uint16_t *x_dev, int M, uint16_t *out_dev, uint16_t *out_normed_dev,
                      void *ws_dev, size_t ws_bytes, moe_stream_t stream)
{
    if (!stack || !x_dev || !out_dev || !aligned16(x_dev) || !aligned16(out_dev)) return MOE_ERR_INVALID_ARG;
    const moe_layer *last = stack->layers[stack->L - 1];
    if (out_normed_dev && !last->ptrs.gamma_next) return MOE_ERR_INVALID_ARG;
    KParams kp;
    int R;
    int rc = prepare(stack->layers[0], M, ws_dev, ws_bytes, kp, R);
    if (rc) return rc;
    bool streamed = false;
    for (int l = 0; l < stack->L; ++l) streamed = streamed || stack->layers[l]->ptrs.slot_of != nullptr;
    if (!streamed && use_grouped(M, R))   // grouped mode, as in moe_decode_layer
        return grouped_forward(stack->layers, stack->L, x_dev, M, out_dev, out_normed_dev, ws_dev, ws_bytes,
                               g_timeout_ns, reinterpret_cast<cudaStream_t>(stream));
    kp.mode = kModeLayers;
    const int H = kp.g.H;
    for (int c0 = 0; c0 < M; c0 += R) {
        const int mc = M - c0 < R ? M - c0 : R;
        if ((rc = plan_for(kp, mc))) return rc;
        for (int l0 = 0; l0 < stack->L; l0 += kMaxLayers) {
            const int nl = stack->L - l0 < kMaxLayers ? stack->L - l0 : kMaxLayers;
            kp.L = nl;
            for (int i = 0; i < nl; ++i) kp.layer[i] = stack->layers[l0 + i]->ptrs;
            kp.x = l0 == 0 ? x_dev + (size_t)c0 * H : out_dev + (size_t)c0 * H;
            kp.out = out_dev + (size_t)c0 * H;
            const bool final_group = l0 + nl == stack->L;
            kp.out_normed = final_group && out_normed_dev ? out_normed_dev + (size_t)c0 * H : nullptr;
            if ((rc = decode_launch(kp, reinterpret_cast<cudaStream_t>(stream)))) return rc;
        }
    }
    return MOE_OK;
}

int moe_stack_forward_host(moe_stack *stack, const uint16_t *x_host, int M, uint16_t *out_host, void *ws_dev,
                           size_t ws_bytes, moe_stream_t stream)
{
    if (!stack || !x_host || !out_host || !ws_dev || M < 1) return MOE_ERR_INVALID_ARG;
    Geo g = stack->layers[0]->geo;
    WsLayout w;
    make_ws_layout(g, M, w);
    if (ws_bytes < w.total) return MOE_ERR_BUFFER_TOO_SMALL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *din = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws_dev) + w.off_stage_in);
    uint16_t *dout = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws_dev) + w.off_stage_out);
    const size_t bytes = (size_t)M * g.H * 2;
    cudaError_t e = cudaMemcpyAsync(din, x_host, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    int rc = moe_stack_forward(stack, din, M, dout, nullptr, ws_dev, ws_bytes, stream);
    if (rc) return rc;
    e = cudaMemcpyAsync(out_host, dout, bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return moe_stream_status(ws_dev, ws_bytes, stream);
}

void moe_stack_destroy(moe_stack *stack)
{
    if (!stack) return;
    free(stack->layers);
    free(stack);
}

int moe_stream_status(void *ws_dev, size_t ws_bytes, moe_stream_t stream)
{
    if (!ws_dev || ws_bytes < (size_t)kCtrlBytes) return MOE_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return check_status_word(ws_dev);
}

}  // extern "C"

namespace {

// Scratch of moe_decode_layer_noalloc: one fixed array per device, shared by
// every call on that device.  Its host-side name is only a handle for the
// runtime; the kernels get the device address looked up below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the array on the current device, looked up once per
// device; the first lookup also zeroes the whole array on `stream` (the
// launch sequence, the status word and every exchanged word start at zero).
int noalloc_scratch(void **out, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    void *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
        if (!p) {
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
            e = cudaMemsetAsync(p, 0, MOE_NOALLOC_SCRATCH_BYTES, stream);
            if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
            g_noalloc_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_decode_layer_noalloc(const moe_layer *layer, const uint16_t *x_dev, int M, uint16_t *out_dev,
                             uint16_t *out_normed_dev, moe_stream_t stream)
{
    if (!layer || M < 1 || !x_dev || !out_dev || !aligned16(x_dev) || !aligned16(out_dev)) return MOE_ERR_INVALID_ARG;
    if (out_normed_dev && !layer->ptrs.gamma_next) return MOE_ERR_INVALID_ARG;
    WsLayout w;
    make_ws_layout_fma(layer->geo, M, w);   // the scratch array holds no grouped-mode regions
    if (w.total > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_BUFFER_TOO_SMALL;
    void *ws = nullptr;
    int rc = noalloc_scratch(&ws, reinterpret_cast<cudaStream_t>(stream));
    if (rc) return rc;
    // the status word is cleared on the stream once every check has passed,
    // just before the first launch
    return decode_layer_impl(layer, x_dev, M, out_dev, out_normed_dev, ws, (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream,
                             false, true);
}

int moe_noalloc_status(moe_stream_t stream)
{
    void *ws = nullptr;
    int rc = noalloc_scratch(&ws, reinterpret_cast<cudaStream_t>(stream));
    if (rc) return rc;
    return moe_stream_status(ws, (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream);
}

int moe_set_grouped(int min_rows)
{
    if (min_rows < 0) return MOE_ERR_INVALID_ARG;
    g_grouped_min_rows = min_rows;
    return MOE_OK;
}

int moe_set_grouped_products(int tensor_cores)
{
    if (tensor_cores != 0 && tensor_cores != 1) return MOE_ERR_INVALID_ARG;
    g_grouped_tc.store(tensor_cores, std::memory_order_relaxed);
    return MOE_OK;
}

int moe_debug_set(int skip_row, long long timeout_ns)
{
    g_skip_row = skip_row;
    g_timeout_ns = timeout_ns > 0 ? timeout_ns : 2000000000LL;
    return MOE_OK;
}

int moe_build_flags(void)
{
#ifdef MOE_DEBUG_BOUNDS
    return MOE_BUILD_DEBUG_BOUNDS;
#else
    return 0;
#endif
}

int moe_debug_inject(int expert)
{
#ifdef MOE_DEBUG_BOUNDS
    g_inject_e = expert < 0 ? -1 : expert;
    return MOE_OK;
#else
    (void)expert;
    return MOE_ERR_UNSUPPORTED;
#endif
}

int moe_debug_trace(void *trace_dev, size_t bytes)
{
    const int sms = device_sms();
    if (trace_dev && (sms <= 0 || bytes < ((size_t)sms * kMaxLayers * kTraceEvents + 2 * kMaxLayers * 16 * 16) * 8))
        return MOE_ERR_BUFFER_TOO_SMALL;
    g_trace = static_cast<unsigned long long *>(trace_dev);
    return MOE_OK;
}

int moe_gate_up_tc(const moe_layer *layer, const float *hn_dev, int M, const int32_t *experts_dev,
                   const uint32_t *masks_dev, int U, float *act_dev, int *err_dev, moe_stream_t stream)
{
    if (!layer || !hn_dev || !experts_dev || !masks_dev || !act_dev || !err_dev || M < 1 || U < 0)
        return MOE_ERR_INVALID_ARG;
    if (layer->ptrs.slot_of) return MOE_ERR_UNSUPPORTED;   // a streamed layer's experts are not at their ids
    if (M > 32 || (2 * layer->geo.I) % 128 != 0 || !bits_ok(layer->geo.rb)) return MOE_ERR_UNSUPPORTED;
    if (U == 0) return MOE_OK;
    return launch_gate_up_tc(*layer, hn_dev, M, experts_dev, masks_dev, U, act_dev, err_dev, g_timeout_ns,
                             reinterpret_cast<cudaStream_t>(stream));
}

int moe_down_tc(const moe_layer *layer, const float *act_dev, int M, const int32_t *experts_dev,
                const uint32_t *masks_dev, int U, float *y_dev, int *err_dev, moe_stream_t stream)
{
    if (!layer || !act_dev || !experts_dev || !masks_dev || !y_dev || !err_dev || M < 1 || U < 0)
        return MOE_ERR_INVALID_ARG;
    if (layer->ptrs.slot_of) return MOE_ERR_UNSUPPORTED;
    if (M > 32 || layer->geo.H % 128 != 0 || !bits_ok(layer->geo.rb)) return MOE_ERR_UNSUPPORTED;
    if (U == 0) return MOE_OK;
    return launch_down_tc(*layer, act_dev, M, experts_dev, masks_dev, U, y_dev, err_dev, g_timeout_ns,
                          reinterpret_cast<cudaStream_t>(stream));
}

namespace {
bool qkv_desc_ok(const moe_qkv_desc &d)
{
    return d.H >= 128 && d.H % kGroup == 0 && d.n_q >= 0 && d.n_k >= 0 && d.n_v >= 0 && d.n_q + d.n_k + d.n_v >= 1 &&
           bits_ok(d.bits) && (long long)d.n_q + d.n_k + d.n_v < (1ll << 30);
}
}  // namespace

int moe_qkv_pack_size(const moe_qkv_desc *desc, size_t *bytes)
{
    if (!desc || !bytes) return MOE_ERR_INVALID_ARG;
    if (!qkv_desc_ok(*desc)) return MOE_ERR_UNSUPPORTED;
    *bytes = (size_t)(desc->n_q + desc->n_k + desc->n_v) * row_bytes(desc->H, desc->bits);
    return MOE_OK;
}

int moe_qkv_pack(const moe_qkv_desc *desc, const moe_src_matrix *q, const moe_src_matrix *k, const moe_src_matrix *v,
                 void *dst_dev, size_t dst_bytes, moe_qkv **out, moe_stream_t stream)
{
    if (!desc || !q || !k || !v || !dst_dev || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!qkv_desc_ok(*desc)) return MOE_ERR_UNSUPPORTED;
    const int rb = row_bytes(desc->H, desc->bits), n = desc->n_q + desc->n_k + desc->n_v;
    if (dst_bytes < (size_t)n * rb) return MOE_ERR_BUFFER_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(dst_dev) & 255) != 0) return MOE_ERR_INVALID_ARG;
    uint8_t *base = static_cast<uint8_t *>(dst_dev);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const moe_src_matrix *src[3] = {q, k, v};
    const int rows[3] = {desc->n_q, desc->n_k, desc->n_v};
    size_t off = 0;
    for (int i = 0; i < 3; ++i) {
        if (rows[i] > 0) {
            const int rc = launch_pack_rows(*src[i], desc->bits, rows[i], desc->H, base + off, st);
            if (rc) return rc;
        }
        off += (size_t)rows[i] * rb;
    }
    moe_qkv *h = static_cast<moe_qkv *>(calloc(1, sizeof(moe_qkv)));
    if (!h) return MOE_ERR_INVALID_ARG;
    h->desc = *desc;
    h->rows = n;
    h->row_bytes = rb;
    h->base = base;
    *out = h;
    return MOE_OK;
}

int moe_qkv_forward(const moe_qkv *qkv, const uint16_t *x_dev, int M, float *y_dev, int *err_dev, moe_stream_t stream)
{
    if (!qkv || !x_dev || !y_dev || !err_dev || M < 1 || !aligned16(x_dev)) return MOE_ERR_INVALID_ARG;
    if ((long long)M * qkv->desc.H > 32768) return MOE_ERR_UNSUPPORTED;
    return launch_qkv(qkv->base, qkv->rows, qkv->desc.H, qkv->desc.bits, x_dev, M, y_dev, err_dev, g_timeout_ns,
                      reinterpret_cast<cudaStream_t>(stream));
}

void moe_qkv_destroy(moe_qkv *qkv) { free(qkv); }

int moe_attn_workspace_size(int T_cap, size_t *bytes)
{
    if (!bytes || T_cap < 1 || T_cap > attn_max_positions()) return MOE_ERR_INVALID_ARG;
    *bytes = attn_workspace_bytes(T_cap);
    return MOE_OK;
}

int moe_attn_decode(const uint16_t *q_dev, const uint16_t *k_cache_dev, const uint16_t *vt_cache_dev, int T_cap,
                    int pos0, int M, float *o_dev, void *ws_dev, size_t ws_bytes, int *err_dev, moe_stream_t stream)
{
    if (!q_dev || !k_cache_dev || !vt_cache_dev || !o_dev || !ws_dev || !err_dev) return MOE_ERR_INVALID_ARG;
    if (M < 1 || M > MOE_ATTN_MAX_ROWS || pos0 < 0 || T_cap < 8 || T_cap % 8 != 0 || pos0 + M > T_cap ||
        T_cap > attn_max_positions())
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_cache_dev) | reinterpret_cast<uintptr_t>(vt_cache_dev) |
         reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(ws_dev)) & 15u)
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < attn_workspace_bytes(T_cap)) return MOE_ERR_BUFFER_TOO_SMALL;
    return launch_attn(q_dev, k_cache_dev, vt_cache_dev, T_cap, pos0, M, o_dev, ws_dev, err_dev, g_timeout_ns,
                       reinterpret_cast<cudaStream_t>(stream));
}

int moe_attn_append(const uint16_t *k_new_dev, const uint16_t *v_new_dev, int M, int pos0, uint16_t *k_cache_dev,
                    uint16_t *vt_cache_dev, int T_cap, moe_stream_t stream)
{
    if (!k_new_dev || !v_new_dev || !k_cache_dev || !vt_cache_dev) return MOE_ERR_INVALID_ARG;
    if (M < 1 || M > MOE_ATTN_MAX_ROWS || pos0 < 0 || T_cap < 1 || pos0 + M > T_cap) return MOE_ERR_INVALID_ARG;
    return launch_attn_append(k_new_dev, v_new_dev, M, pos0, k_cache_dev, vt_cache_dev, T_cap,
                              reinterpret_cast<cudaStream_t>(stream));
}

const char *moe_status_str(int status)
{
    switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_BUFFER_TOO_SMALL: return "MOE_ERR_BUFFER_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    case MOE_ERR_NOT_RESIDENT: return "MOE_ERR_NOT_RESIDENT";
    default: return "MOE_ERR_UNKNOWN";
    }
}

int moe_last_cuda_error(void) { return t_last_cuda_error; }

long long moe_launch_count(int reset)
{
    const long long n = t_launches;
    if (reset) t_launches = 0;
    return n;
}

int moe_selftest_host(void) { return unpack_selftest_host() + plan_selftest_host() + ws_layout_selftest_host(); }

}  // extern "C"
