// Streamed layers: the routed experts of a layer live in host memory (on
// GB300, the Grace side, reached over NVLink-C2C), and only the experts the
// router selects are copied into an HBM cache of expert slots, the GB300
// counterpart of the pages' SSD expert streaming (flash-moe, "SSD Expert
// Streaming": only the selected experts are loaded, and a cache managed
// least-recently-used keeps the popular ones; AiiStream Q3.6 article: the
// next layer's experts are predicted and loaded ahead; "Qwen3.5-397B on M5
// Max", temporal expert prediction).
//
// The router, the norm weights and the shared expert stay resident in HBM.
// The decode kernel is the resident one: its routing warp replaces each
// selected expert id by the expert's cache slot (the layer's slot map), so
// the expert rows are read from the cache with the same address arithmetic
// and the results are bitwise those of the resident layer.  An expert with
// no slot is reported (MOE_ERR_NOT_RESIDENT), never read past the cache.
//
// The host side here keeps, per layer, the slot of every expert (a host
// mirror of the device slot map), the expert held by every slot and a use
// stamp per slot (least recently used evicted first), and fetches missing
// experts (each expert's gate/up units and its down rows are contiguous in
// the packed blob): with pinned host memory, one gather kernel reads them
// all over the host link (about 200 GB/s measured on GB300, against about
// 150 for copy-engine copies of expert-sized pieces); otherwise one copy per
// piece.
// moe_streamed_forward runs a token through a stack of such layers: route
// layer l, copy its missing experts, decode it; with prediction, layer
// l + 1's router also runs on layer l's input, and the experts it names are
// copied on a second stream while layer l is decoded.  (Both routers run on
// the caller's stream: the decode kernel is a cooperative launch over every
// SM, and nothing of this runtime runs kernels beside it; only copies
// overlap it.)
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "moe_internal.h"

struct moe_streamed {
    moe_layer layer;                 // resident parts and cache in dev_buf; ptrs.slot_of set
    const uint8_t *host;             // the whole packed blob, host memory
    size_t off_cache_gu, off_cache_down, off_shared, off_map, off_jobs;
    bool host_mapped;                // the device can read `host` directly (pinned host memory)
    int n_slots;
    int32_t *slot_of_dev;
    std::vector<int32_t> slot_of;    // expert -> slot, or -1
    std::vector<int32_t> owner;      // slot -> expert, or -1
    std::vector<uint64_t> stamp;     // last use of a slot
    uint64_t tick;
    long long hits, misses, fetched, bytes, predicted, predicted_used;
    std::vector<int32_t> last_pred;  // the experts last predicted for this layer
    bool prefetch_pending;           // copies of a prefetch into this cache are in flight (copy stream)
    cudaEvent_t ev_prefetched, ev_used;
};

namespace moe {
namespace {

struct StreamedLayout {
    size_t cache_gu, cache_down, shared, map, jobs, total;
};

// One copy of the gather kernel: n16 16-byte words from src (host memory
// the device can read) to dst (device memory).
struct CopyJob {
    const uint4 *src;
    uint4 *dst;
    unsigned long long n16;
    unsigned long long pad;
};
constexpr int kGatherCtasPerJob = 16;

// The experts' rows from host memory into their cache slots: CTA (x, j)
// takes every gridDim.x-th stretch of job j, four 16-byte loads in flight
// per thread (the host link is latency-bound otherwise); loads bypass L1.
__global__ void __launch_bounds__(256) gather_kernel(const CopyJob *jobs)
{
    const CopyJob j = jobs[blockIdx.y];
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 1
    for (; i + 3 * stride < j.n16; i += 4 * stride) {
        const uint4 a = __ldcs(j.src + i), b = __ldcs(j.src + i + stride), c = __ldcs(j.src + i + 2 * stride),
                    d = __ldcs(j.src + i + 3 * stride);
        j.dst[i] = a;
        j.dst[i + stride] = b;
        j.dst[i + 2 * stride] = c;
        j.dst[i + 3 * stride] = d;
    }
#pragma unroll 1
    for (; i < j.n16; i += stride) j.dst[i] = __ldcs(j.src + i);
}

StreamedLayout streamed_layout(const Geo &g, int n_slots)
{
    StreamedLayout s;
    size_t o = align_up(g.off_gu, 256);   // router (both copies), gamma, gamma_next at their blob offsets
    s.cache_gu = o;
    o = align_up(o + (size_t)n_slots * g.I * 2 * g.g_bytes, 256);
    s.cache_down = o;
    o = align_up(o + (size_t)n_slots * g.H * g.d_bytes, 256);
    s.shared = o;
    o = align_up(o + (g.total - g.off_sgu), 256);
    s.map = o;
    o = align_up(o + (size_t)g.E * 4, 256);
    s.jobs = o;
    o = align_up(o + (size_t)2 * n_slots * sizeof(CopyJob), 256);
    s.total = o;
    return s;
}

int cuda_fail(cudaError_t e)
{
    note_cuda_error((int)e);
    return MOE_ERR_CUDA;
}

size_t expert_gu_bytes(const Geo &g) { return (size_t)g.I * 2 * g.g_bytes; }
size_t expert_down_bytes(const Geo &g) { return (size_t)g.H * g.d_bytes; }

// Makes experts ids[0 .. n) resident (each distinct id once), copying the
// missing ones on `st`, least recently used slots first and never a slot
// that holds one of ids.  Counts hits and misses when `count` is set.
int make_resident(moe_streamed *s, const int32_t *ids, int n, cudaStream_t st, bool count, int *fetched_out)
{
    const Geo &g = s->layer.geo;
    const uint64_t now = ++s->tick;
    std::vector<int32_t> want;
    want.reserve(n);
    for (int i = 0; i < n; ++i) {
        const int e = ids[i];
        if (e < 0 || e >= g.E) return MOE_ERR_INVALID_ARG;
        bool dup = false;
        for (int w : want) dup = dup || w == e;
        if (!dup) want.push_back(e);
    }
    if ((int)want.size() > s->n_slots) return MOE_ERR_BUFFER_TOO_SMALL;
    // stamp the residents first so that none of them is evicted below
    for (int e : want)
        if (s->slot_of[e] >= 0) s->stamp[s->slot_of[e]] = now;
    int fetched = 0;
    bool changed = false;
    std::vector<CopyJob> jobs;
    uint8_t *dev = s->layer.base;
    for (int e : want) {
        if (s->slot_of[e] >= 0) {
            if (count) ++s->hits;
            continue;
        }
        if (count) ++s->misses;
        int victim = -1;
        for (int c = 0; c < s->n_slots; ++c)
            if (s->stamp[c] != now && (victim < 0 || s->stamp[c] < s->stamp[victim])) victim = c;
        if (victim < 0) return MOE_ERR_BUFFER_TOO_SMALL;
        if (s->owner[victim] >= 0) s->slot_of[s->owner[victim]] = -1;
        uint8_t *dgu = dev + s->off_cache_gu + (size_t)victim * expert_gu_bytes(g);
        uint8_t *ddn = dev + s->off_cache_down + (size_t)victim * expert_down_bytes(g);
        const uint8_t *hgu = s->host + g.off_gu + (size_t)e * expert_gu_bytes(g);
        const uint8_t *hdn = s->host + g.off_down + (size_t)e * expert_down_bytes(g);
        if (s->host_mapped) {
            jobs.push_back({reinterpret_cast<const uint4 *>(hgu), reinterpret_cast<uint4 *>(dgu), expert_gu_bytes(g) / 16, 0});
            jobs.push_back({reinterpret_cast<const uint4 *>(hdn), reinterpret_cast<uint4 *>(ddn), expert_down_bytes(g) / 16, 0});
        } else {
            cudaError_t err = cudaMemcpyAsync(dgu, hgu, expert_gu_bytes(g), cudaMemcpyHostToDevice, st);
            if (err == cudaSuccess) err = cudaMemcpyAsync(ddn, hdn, expert_down_bytes(g), cudaMemcpyHostToDevice, st);
            if (err != cudaSuccess) return cuda_fail(err);
        }
        s->owner[victim] = e;
        s->slot_of[e] = victim;
        s->stamp[victim] = now;
        s->bytes += (long long)(expert_gu_bytes(g) + expert_down_bytes(g));
        ++s->fetched;
        ++fetched;
        changed = true;
    }
    if (!jobs.empty()) {
        // one launch reads every missing expert over the host link (the job
        // table's pageable source is staged before the call returns)
        CopyJob *jd = reinterpret_cast<CopyJob *>(dev + s->off_jobs);
        cudaError_t err = cudaMemcpyAsync(jd, jobs.data(), jobs.size() * sizeof(CopyJob), cudaMemcpyHostToDevice, st);
        if (err != cudaSuccess) return cuda_fail(err);
        gather_kernel<<<dim3(kGatherCtasPerJob, (unsigned)jobs.size()), 256, 0, st>>>(jd);
        note_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return cuda_fail(err);
    }
    if (changed) {
        // pageable source: the runtime stages it before returning, so the
        // mirror may change right after
        const cudaError_t err = cudaMemcpyAsync(s->slot_of_dev, s->slot_of.data(), (size_t)g.E * 4,
                                                cudaMemcpyHostToDevice, st);
        if (err != cudaSuccess) return cuda_fail(err);
    }
    if (fetched_out) *fetched_out = fetched;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_streamed_size(const moe_layer_desc *desc, int n_slots, size_t *dev_bytes)
{
    if (!desc || !dev_bytes || n_slots < 1) return MOE_ERR_INVALID_ARG;
    Geo g;
    if (!make_geo(*desc, g)) return MOE_ERR_UNSUPPORTED;
    if (n_slots < g.k || n_slots > g.E) return MOE_ERR_INVALID_ARG;
    *dev_bytes = streamed_layout(g, n_slots).total;
    return MOE_OK;
}

int moe_streamed_create(const moe_layer *packed, void *host_blob, size_t host_bytes, void *dev_buf, size_t dev_bytes,
                        int n_slots, moe_streamed **out, moe_stream_t stream)
{
    if (!packed || !host_blob || !dev_buf || !out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (packed->ptrs.slot_of) return MOE_ERR_INVALID_ARG;
    const Geo &g = packed->geo;
    if (n_slots < g.k || n_slots > g.E) return MOE_ERR_INVALID_ARG;
    if (host_bytes < g.total) return MOE_ERR_BUFFER_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(dev_buf) & 255) != 0) return MOE_ERR_INVALID_ARG;
    const StreamedLayout sl = streamed_layout(g, n_slots);
    if (dev_bytes < sl.total) return MOE_ERR_BUFFER_TOO_SMALL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    moe_streamed *s = new (std::nothrow) moe_streamed();
    if (!s) return MOE_ERR_INVALID_ARG;
    uint8_t *dev = static_cast<uint8_t *>(dev_buf);
    s->host = static_cast<const uint8_t *>(host_blob);
    s->off_cache_gu = sl.cache_gu;
    s->off_cache_down = sl.cache_down;
    s->off_shared = sl.shared;
    s->off_map = sl.map;
    s->off_jobs = sl.jobs;
    s->n_slots = n_slots;
    {
        // pinned (or registered) host memory is read by the gather kernel;
        // any other host memory goes through copies
        cudaPointerAttributes pa;
        s->host_mapped = cudaPointerGetAttributes(&pa, host_blob) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
                         pa.devicePointer == host_blob && (reinterpret_cast<uintptr_t>(host_blob) & 15) == 0;
        cudaGetLastError();
    }
    s->slot_of.assign(g.E, -1);
    s->owner.assign(n_slots, -1);
    s->stamp.assign(n_slots, 0);
    s->slot_of_dev = reinterpret_cast<int32_t *>(dev + sl.map);
    // the whole blob to host memory; the resident parts (router, gammas,
    // shared expert) to the device buffer; an empty cache and slot map
    cudaError_t err = cudaMemcpyAsync(host_blob, packed->base, g.total, cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaMemcpyAsync(dev, packed->base, g.off_gu, cudaMemcpyDeviceToDevice, st);
    if (err == cudaSuccess && g.total > g.off_sgu)
        err = cudaMemcpyAsync(dev + sl.shared, packed->base + g.off_sgu, g.total - g.off_sgu, cudaMemcpyDeviceToDevice,
                              st);
    if (err == cudaSuccess) err = cudaMemsetAsync(dev + sl.cache_gu, 0, sl.shared - sl.cache_gu, st);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(s->slot_of_dev, s->slot_of.data(), (size_t)g.E * 4, cudaMemcpyHostToDevice, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&s->ev_prefetched, cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&s->ev_used, cudaEventDisableTiming);
    if (err != cudaSuccess) {
        delete s;
        return cuda_fail(err);
    }
    s->layer.desc = packed->desc;
    s->layer.geo = g;
    s->layer.base = dev;
    s->layer.bytes = dev_bytes;
    LayerPtrs &p = s->layer.ptrs;
    p.router = dev + g.off_router;
    p.router_t = dev + g.off_router_t;
    p.gamma = reinterpret_cast<const uint16_t *>(dev + g.off_gamma);
    p.gamma_next = packed->ptrs.gamma_next ? reinterpret_cast<const uint16_t *>(dev + g.off_gamma_next) : nullptr;
    p.gu = dev + sl.cache_gu;
    p.down = dev + sl.cache_down;
    p.sgu = g.has_shared ? dev + sl.shared : nullptr;
    p.sdown = g.has_shared ? dev + sl.shared + (g.off_sdown - g.off_sgu) : nullptr;
    p.slot_of = s->slot_of_dev;
    p.n_slots = n_slots;
    *out = s;
    return MOE_OK;
}

const moe_layer *moe_streamed_layer(const moe_streamed *s) { return s ? &s->layer : nullptr; }

int moe_streamed_prepare(moe_streamed *s, const int32_t *expert_ids, int n, moe_stream_t stream, int *fetched)
{
    if (!s || (!expert_ids && n > 0) || n < 0) return MOE_ERR_INVALID_ARG;
    return make_resident(s, expert_ids, n, reinterpret_cast<cudaStream_t>(stream), true, fetched);
}

int moe_streamed_stats(const moe_streamed *s, long long *hits, long long *misses, long long *fetched,
                       long long *bytes, long long *predicted, long long *predicted_used)
{
    if (!s) return MOE_ERR_INVALID_ARG;
    if (hits) *hits = s->hits;
    if (misses) *misses = s->misses;
    if (fetched) *fetched = s->fetched;
    if (bytes) *bytes = s->bytes;
    if (predicted) *predicted = s->predicted;
    if (predicted_used) *predicted_used = s->predicted_used;
    return MOE_OK;
}

void moe_streamed_destroy(moe_streamed *s)
{
    if (!s) return;
    cudaEventDestroy(s->ev_prefetched);
    cudaEventDestroy(s->ev_used);
    delete s;
}

int moe_streamed_forward(moe_streamed *const *layers, int L, const uint16_t *x_dev, int M, uint16_t *out_dev,
                         uint16_t *out_normed_dev, void *ws_dev, size_t ws_bytes, void *route_dev, size_t route_bytes,
                         int predict, moe_stream_t stream, moe_stream_t copy_stream)
{
    if (!layers || L < 1 || !x_dev || !out_dev || !ws_dev || !route_dev || M < 1) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < L; ++l)
        if (!layers[l]) return MOE_ERR_INVALID_ARG;
    const Geo &g0 = layers[0]->layer.geo;
    for (int l = 1; l < L; ++l)
        if (layers[l]->layer.geo.H != g0.H || layers[l]->layer.geo.k != g0.k) return MOE_ERR_INVALID_ARG;
    if (M > rows_per_launch(g0.H)) return MOE_ERR_UNSUPPORTED;   // one persistent launch per layer
    const int nk = M * g0.k;
    if (route_bytes < (size_t)nk * 16) return MOE_ERR_BUFFER_TOO_SMALL;
    if (predict && !copy_stream) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);
    int32_t *ids = static_cast<int32_t *>(route_dev);
    float *w = reinterpret_cast<float *>(ids + 2 * nk);
    std::vector<int32_t> h_ids(2 * nk);   // layer l's routing, then the prediction of layer l + 1
    cudaError_t err = cudaSuccess;
    int rc = MOE_OK;
    for (int l = 0; l < L && rc == MOE_OK; ++l) {
        moe_streamed *s = layers[l];
        const uint16_t *in = l == 0 ? x_dev : out_dev;
        const bool pred = predict && l + 1 < L;
        // route layer l on its input; as the prediction of layer l + 1, its
        // router on the same input (both on this stream, one host wait)
        if ((rc = moe_router_topk(&s->layer, in, M, ids, w, ws_dev, ws_bytes, stream))) break;
        if (pred && (rc = moe_router_topk(&layers[l + 1]->layer, in, M, ids + nk, w + nk, ws_dev, ws_bytes, stream)))
            break;
        if ((err = cudaMemcpyAsync(h_ids.data(), ids, (size_t)(pred ? 2 : 1) * nk * 4, cudaMemcpyDeviceToHost, st)) !=
                cudaSuccess ||
            (err = cudaStreamSynchronize(st)) != cudaSuccess) {
            rc = cuda_fail(err);
            break;
        }
        // how many of layer l's experts its prediction named
        if (!s->last_pred.empty()) {
            for (int i = 0; i < nk; ++i) {
                bool in_pred = false;
                for (int e : s->last_pred) in_pred = in_pred || e == h_ids[i];
                s->predicted_used += in_pred ? 1 : 0;
            }
            s->last_pred.clear();
        }
        // layer l's prefetch (issued one layer earlier) lands first, then the
        // experts it still misses are copied on this stream
        if (s->prefetch_pending) {
            if ((err = cudaStreamWaitEvent(st, s->ev_prefetched, 0)) != cudaSuccess) {
                rc = cuda_fail(err);
                break;
            }
            s->prefetch_pending = false;
        }
        if ((rc = make_resident(s, h_ids.data(), nk, st, true, nullptr))) break;
        // prefetch of layer l + 1 on the copy stream, after the last decode
        // that read its cache; it overlaps the decode of layer l
        if (pred) {
            moe_streamed *n = layers[l + 1];
            if ((err = cudaStreamWaitEvent(cs, n->ev_used, 0)) != cudaSuccess) {
                rc = cuda_fail(err);
                break;
            }
            n->predicted += nk;
            n->last_pred.assign(h_ids.begin() + nk, h_ids.begin() + 2 * nk);
            if ((rc = make_resident(n, h_ids.data() + nk, nk, cs, false, nullptr))) break;
            if ((err = cudaEventRecord(n->ev_prefetched, cs)) != cudaSuccess) {
                rc = cuda_fail(err);
                break;
            }
            n->prefetch_pending = true;
        }
        uint16_t *o_n = l == L - 1 ? out_normed_dev : nullptr;
        if ((rc = moe_decode_layer(&s->layer, in, M, out_dev, o_n, ws_dev, ws_bytes, stream))) break;
        if ((err = cudaEventRecord(s->ev_used, st)) != cudaSuccess) {
            rc = cuda_fail(err);
            break;
        }
    }
    return rc;
}

}  // extern "C"
