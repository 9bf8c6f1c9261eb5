// Grouped mode: layers over more token rows than one persistent launch holds
// (M above rows_per_launch).  Up to 32 rows go through a layer together, so
// each selected expert is read once for all of them (PureDrive-35B-A3B model
// card, "How it works": the weights are read once for all verify rows), and
// the expert products run on the tensor cores (moe_tc.cu) where rows per
// expert make them a real contraction.
//
// Per layer and group of rows:
//   1. rms_sigma_kernel: hn rows (fp32) and the shared-expert gate sigma;
//   2. router_kernel + topk_kernel: fp32 router logits (FMA pipes), the warp
//      top-k per row (ties to the lower id) and the renormalised softmax
//      weights;
//   3. group_kernel: distinct experts in id order with their row masks;
//   4. tensor-core gate/up + SwiGLU, then down, for the routed experts
//      (slot count read on the device) and the shared expert, one launch per
//      projection;
//   5. combine_kernel: out = bf16(x + sum_i w_i y_i + sigma y_s) in expert-id
//      order, and the fused next RMSNorm when asked for.
// The expert products carry the tensor cores' accumulation error (see
// moe_tc.cu), so values are not row-exact; routing decisions are those of the
// oracle wherever the top-k logit gap exceeds the fp32 rounding of the logits.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float bf2f_g(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf_g(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    return t;
}

// Code h of a packed row's LSB-first stream at `bits` bits.
__device__ __forceinline__ uint32_t code_of(const uint8_t *row, int h, int bits)
{
    const int bit = h * bits, byte = bit >> 3, off = bit & 7;
    const uint32_t v = (uint32_t)row[byte] | ((uint32_t)row[byte + 1] << 8);
    return (v >> off) & ((1u << bits) - 1u);
}

// One CTA per row: hn = x rsqrt(mean(x^2) + eps) gamma (fp32), and sigma =
// sigmoid(w_sg . hn) from the router's last row when there is a shared expert.
__global__ void __launch_bounds__(kRowThreads) rms_sigma_kernel(const uint16_t *__restrict__ x, int H,
                                                                 const uint16_t *__restrict__ gamma, float eps,
                                                                 const uint8_t *__restrict__ sgate_row, int qb,
                                                                 float *__restrict__ hn, float *__restrict__ sigma)
{
    __shared__ float red[kRowThreads / 32];
    const int m = blockIdx.x;
    const uint16_t *xr = x + (size_t)m * H;
    float ss = 0.f;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float v = bf2f_g(xr[h]);
        ss = fmaf(v, v, ss);
    }
    const float rinv = rsqrtf(block_sum(ss, red) / (float)H + eps);
    float dot = 0.f;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float v = bf2f_g(xr[h]) * rinv * bf2f_g(gamma[h]);
        hn[(size_t)m * H + h] = v;
        if (sgate_row) {
            float w;
            if (qb == 0) {
                w = reinterpret_cast<const float *>(sgate_row)[h];
            } else {
                const uint32_t sb = reinterpret_cast<const uint32_t *>(sgate_row + (size_t)H * qb / 8)[h / kGroup];
                w = fmaf((float)code_of(sgate_row, h, qb), __uint_as_float(sb << 16), __uint_as_float(sb & 0xFFFF0000u));
            }
            dot = fmaf(w, v, dot);
        }
    }
    if (sgate_row) {
        const float t = block_sum(dot, red);
        if (threadIdx.x == 0) sigma[m] = 1.0f / (1.0f + expf(-t));
    } else if (threadIdx.x == 0) {
        sigma[m] = 0.f;
    }
}

// Router logits of M rows: one CTA per expert row e; the row is dequantised
// into shared memory (w = q s + b per group of 64, or fp32), then warp w
// takes token rows w, w + 8, ... with lane l summing inputs l, l + 32, ...
// in fp32, and a butterfly over the lanes.  logits [M][E].
__global__ void __launch_bounds__(kRowThreads) router_kernel(const uint8_t *__restrict__ router, int rr_bytes, int qb,
                                                              int H, int E, const float *__restrict__ hn, int M,
                                                              float *__restrict__ logits)
{
    extern __shared__ float wrow[];
    const int e = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint8_t *row = router + (size_t)e * rr_bytes;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        if (qb == 0) {
            wrow[h] = reinterpret_cast<const float *>(row)[h];
        } else {
            const uint32_t sb = reinterpret_cast<const uint32_t *>(row + (size_t)H * qb / 8)[h / kGroup];
            wrow[h] = fmaf((float)code_of(row, h, qb), __uint_as_float(sb << 16), __uint_as_float(sb & 0xFFFF0000u));
        }
    }
    __syncthreads();
    for (int m = warp; m < M; m += kRowThreads / 32) {
        const float *x = hn + (size_t)m * H;
        float acc = 0.f;
        for (int h = lane; h < H; h += 32) acc = fmaf(wrow[h], x[h], acc);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0) logits[(size_t)m * E + e] = acc;
    }
}

// Top-k of each row's logits, one warp per row (E <= 512: up to 16 per
// lane): k rounds of the warp-wide largest remaining logit, exact ties to the
// lower expert id; then the softmax over the kept k (the full softmax's
// probabilities divided by their top-k sum).  idx, w [M][k] in selection order.
__global__ void __launch_bounds__(32) topk_kernel(const float *__restrict__ logits, int E, int k,
                                                  int32_t *__restrict__ idx, float *__restrict__ w)
{
    const int m = blockIdx.x, lane = threadIdx.x;
    constexpr int NPL = kMaxE / 32;
    float v[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? logits[(size_t)m * E + e] : -INFINITY;
    }
    float top0 = 0.f, mine = 0.f;
    int mine_e = -1;
    for (int r = 0; r < k; ++r) {
        // the lane's best (largest value, lowest index on ties)
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && (v[i] > bv || (v[i] == bv && e < be))) { bv = v[i]; be = e; }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        if (r == 0) top0 = bv;
        if ((be & 31) == lane) {
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (lane + 32 * i == be) v[i] = -INFINITY;
        }
        if (lane == r) { mine = bv; mine_e = be; }
    }
    const float ev = lane < k ? expf(mine - top0) : 0.f;
    float z = ev;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    if (lane < k) {
        idx[m * k + lane] = mine_e;
        w[m * k + lane] = ev / z;
    }
}

// One CTA: the distinct experts of M rows' top-k choices in id order, the
// row mask of each, the slot of each (row, choice), the slot count, and at
// entry shared_pos the shared expert's single slot (expert 0 of the shared
// weights, every row).
__global__ void __launch_bounds__(1024) group_kernel(const int32_t *__restrict__ idx, int M, int k, int E,
                                                     int shared_pos, int32_t *__restrict__ experts,
                                                     uint32_t *__restrict__ masks, int *__restrict__ count,
                                                     int32_t *__restrict__ slotof)
{
    __shared__ uint32_t emask[kMaxE];
    __shared__ int eslot[kMaxE];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) emask[e] = 0u;
    __syncthreads();
    for (int t = tid; t < M * k; t += blockDim.x) {
        const int e = idx[t];
        if (e >= 0 && e < E) atomicOr(&emask[e], 1u << (t / k));
    }
    __syncthreads();
    if (tid < 32) {
        int U = 0;
        for (int c0 = 0; c0 < E; c0 += 32) {
            const int e = c0 + tid;
            const uint32_t em = e < E ? emask[e] : 0u;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, em != 0u);
            if (em) {
                const int pos = U + __popc(bal & ((1u << tid) - 1u));
                experts[pos] = e;
                masks[pos] = em;
                eslot[e] = pos;
            }
            U += __popc(bal);
        }
        if (tid == 0) {
            *count = U;
            experts[shared_pos] = 0;
            masks[shared_pos] = M >= 32 ? 0xFFFFFFFFu : ((1u << M) - 1u);
        }
    }
    __syncthreads();
    for (int t = tid; t < M * k; t += blockDim.x) {
        const int e = idx[t];
        slotof[t] = (e >= 0 && e < E) ? eslot[e] : 0;
    }
}

// CTA (m, part): out = bf16(x + sum_i w_i y[slot_i] + sigma y_s) for row m,
// outputs part * H / gridDim.y .. (the choices summed in expert-id order);
// then, with one part per row, if asked, out_n = bf16(RMSNorm(bf16 out)
// gamma_next).  x and out may alias.
__global__ void __launch_bounds__(kRowThreads) combine_kernel(
    const uint16_t *x, int H, int M, int k, const float *__restrict__ w, const int32_t *__restrict__ slotof,
    const float *__restrict__ y, const float *__restrict__ ysh, const float *__restrict__ sigma,
    const uint16_t *__restrict__ gamma_next, float eps, uint16_t *out, uint16_t *__restrict__ out_n)
{
    __shared__ float red[kRowThreads / 32];
    __shared__ int os[kMaxK];
    __shared__ float ow[kMaxK];
    const int m = blockIdx.x;
    if (threadIdx.x == 0) {
        // slots are numbered in expert-id order: sort the row's choices by slot
        for (int i = 0; i < k; ++i) {
            int s = slotof[m * k + i];
            float wv = w[m * k + i];
            int j = i;
            for (; j > 0 && os[j - 1] > s; --j) { os[j] = os[j - 1]; ow[j] = ow[j - 1]; }
            os[j] = s;
            ow[j] = wv;
        }
    }
    __syncthreads();
    const float sg = sigma[m];
    float ss = 0.f;
    // a grid of several CTAs per row (no out_n) splits the row's H outputs
    const int hs = H / (int)gridDim.y, h0 = hs * (int)blockIdx.y, h1 = h0 + hs;
    for (int h = h0 + threadIdx.x; h < h1; h += blockDim.x) {
        float acc = 0.f;
        for (int i = 0; i < k; ++i) acc = fmaf(ow[i], y[((size_t)os[i] * M + m) * H + h], acc);
        if (ysh) acc = fmaf(sg, ysh[(size_t)m * H + h], acc);
        const uint16_t o = f2bf_g(bf2f_g(x[(size_t)m * H + h]) + acc);
        out[(size_t)m * H + h] = o;
        const float of = bf2f_g(o);
        ss = fmaf(of, of, ss);
    }
    if (!out_n) return;
    const float rinv = rsqrtf(block_sum(ss, red) / (float)H + eps);
    for (int h = threadIdx.x; h < H; h += blockDim.x)
        out_n[(size_t)m * H + h] = f2bf_g(bf2f_g(out[(size_t)m * H + h]) * rinv * bf2f_g(gamma_next[h]));
}

int check_launch()
{
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        note_cuda_error((int)e);
        return MOE_ERR_CUDA;
    }
    note_launch();
    return MOE_OK;
}

}  // namespace

// One layer over mg <= kGroupRows rows of x (bf16 [mg][H]) into out (and
// out_n when not NULL).  ws / w: the caller's workspace and its layout for
// the call's M.
int grouped_layer(const moe_layer &L, const uint16_t *x, int mg, uint16_t *out, uint16_t *out_n, uint8_t *ws,
                  size_t ws_bytes, const WsLayout &w, long long timeout_ns, cudaStream_t st)
{
    const Geo &g = L.geo;
    int32_t *idx = reinterpret_cast<int32_t *>(ws + w.off_g_idx);
    float *wt = reinterpret_cast<float *>(ws + w.off_g_w);
    float *hn = reinterpret_cast<float *>(ws + w.off_g_hn);
    float *sigma = reinterpret_cast<float *>(ws + w.off_g_sigma);
    int32_t *slotof = reinterpret_cast<int32_t *>(ws + w.off_g_slotof);
    int32_t *experts = reinterpret_cast<int32_t *>(ws + w.off_g_experts);
    uint32_t *masks = reinterpret_cast<uint32_t *>(ws + w.off_g_masks);
    int *count = reinterpret_cast<int *>(ws + w.off_g_count);
    float *act = reinterpret_cast<float *>(ws + w.off_g_act);
    float *act_s = reinterpret_cast<float *>(ws + w.off_g_act_s);
    float *y = reinterpret_cast<float *>(ws + w.off_g_y);
    float *ysh = reinterpret_cast<float *>(ws + w.off_g_ysh);
    int *err = &reinterpret_cast<Ctrl *>(ws)->status;
    const int Umax = g.E < mg * g.k ? g.E : mg * g.k;
    int rc;
    const uint8_t *sgate_row = g.has_shared ? L.ptrs.router + (size_t)g.E * g.rr_bytes : nullptr;
    rms_sigma_kernel<<<mg, kRowThreads, 0, st>>>(x, g.H, L.ptrs.gamma, g.eps, sgate_row, g.qb, hn, sigma);
    if ((rc = check_launch())) return rc;
    // routing: fp32 logits (into the routed-output buffer, free until the down
    // projection), then the warp top-k per row
    float *logits = y;
    router_kernel<<<g.E, kRowThreads, (size_t)g.H * 4, st>>>(L.ptrs.router, g.rr_bytes, g.qb, g.H, g.E, hn, mg,
                                                                 logits);
    if ((rc = check_launch())) return rc;
    topk_kernel<<<mg, 32, 0, st>>>(logits, g.E, g.k, idx, wt);
    if ((rc = check_launch())) return rc;
    group_kernel<<<1, 1024, 0, st>>>(idx, mg, g.k, g.E, w.grp_slots, experts, masks, count, slotof);
    if ((rc = check_launch())) return rc;
    // routed experts (set a, slot count on the device) and the shared expert
    // (set b: its own weights, the one slot at entry grp_slots) in one launch
    // per projection, so the shared expert's few tiles run beside the routed
    // ones instead of after them
    const int32_t *she = experts + w.grp_slots;
    const uint32_t *shm = masks + w.grp_slots;
    const TcSetHost gu_r{L.ptrs.gu, 2 * g.I, g.H, g.g_bytes, hn, 0, experts, masks, count, act};
    const TcSetHost gu_s{L.ptrs.sgu, 2 * g.Is, g.H, g.sg_bytes, hn, 0, she, shm, nullptr, act_s};
    const TcSetHost dn_r{L.ptrs.down, g.H, g.I, g.d_bytes, act, mg, experts, masks, count, y};
    const TcSetHost dn_s{L.ptrs.sdown, g.H, g.Is, g.sd_bytes, act_s, mg, she, shm, nullptr, ysh};
    // the FMA products (each slot's rows read once, one pass per token row of
    // the slot) unless the tensor-core products are asked for or the widths
    // exceed the one-vector kernel's
    if (!grouped_products_tc() && g.H <= 2048 && g.I <= 2048 && g.H % 128 == 0 && g.I % 128 == 0 &&
        (!g.has_shared || g.Is % 128 == 0)) {
        const TcSetHost *gs = g.has_shared ? &gu_s : nullptr;
        const TcSetHost *ds = g.has_shared ? &dn_s : nullptr;
        if ((rc = launch_grouped_fma(true, g.rb, gu_r, Umax, g.sb, gs, 1, mg, err, timeout_ns, st))) return rc;
        if ((rc = launch_grouped_fma(false, g.rb, dn_r, Umax, g.sb, ds, 1, mg, err, timeout_ns, st))) return rc;
    } else {
    const bool fused = g.has_shared && (g.sb == g.rb || g.sb == 8);
    if ((rc = launch_grouped_tc2(true, g.rb, gu_r, Umax, g.sb, fused ? &gu_s : nullptr, 1, mg, err, timeout_ns, st)))
        return rc;
    if (g.has_shared && !fused &&
        (rc = launch_grouped_tc2(true, g.sb, gu_s, 1, g.sb, nullptr, 0, mg, err, timeout_ns, st)))
        return rc;
    if ((rc = launch_grouped_tc2(false, g.rb, dn_r, Umax, g.sb, fused ? &dn_s : nullptr, 1, mg, err, timeout_ns, st)))
        return rc;
    if (g.has_shared && !fused &&
        (rc = launch_grouped_tc2(false, g.sb, dn_s, 1, g.sb, nullptr, 0, mg, err, timeout_ns, st)))
        return rc;
    }
    // without the fused RMSNorm, 8 CTAs per row (each a whole number of 256-wide parts)
    const int parts = (!out_n && g.H % (8 * kRowThreads) == 0) ? 8 : 1;
    combine_kernel<<<dim3((unsigned)mg, (unsigned)parts), kRowThreads, 0, st>>>(
        x, g.H, mg, g.k, wt, slotof, y, g.has_shared ? ysh : nullptr, sigma, L.ptrs.gamma_next, g.eps, out, out_n);
    return check_launch();
}

// M rows (any M) through L layers in grouped mode, kGroupRows rows at a
// time: x -> out (bf16 [M][H]); out_n (if not NULL) after the last layer.
int grouped_forward(const moe_layer *const *layers, int L, const uint16_t *x, int M, uint16_t *out, uint16_t *out_n,
                    void *ws_dev, size_t ws_bytes, long long timeout_ns, cudaStream_t st)
{
    const Geo &g = layers[0]->geo;
    WsLayout w;
    make_ws_layout(g, M, w);
    if (ws_bytes < w.total || w.grp_rows == 0) return MOE_ERR_BUFFER_TOO_SMALL;
    if ((2 * g.I) % 128 || g.H % 128 || (g.has_shared && (2 * g.Is) % 128)) return MOE_ERR_UNSUPPORTED;
    uint8_t *ws = static_cast<uint8_t *>(ws_dev);
    uint16_t *ping[2] = {reinterpret_cast<uint16_t *>(ws + w.off_g_ping),
                         reinterpret_cast<uint16_t *>(ws + w.off_g_ping) + (size_t)w.grp_rows * g.H};
    for (int r0 = 0; r0 < M; r0 += w.grp_rows) {
        const int mg = M - r0 < w.grp_rows ? M - r0 : w.grp_rows;
        const uint16_t *cur = x + (size_t)r0 * g.H;
        for (int l = 0; l < L; ++l) {
            const bool last = l == L - 1;
            uint16_t *dst = last ? out + (size_t)r0 * g.H : ping[l & 1];
            uint16_t *dn = last && out_n ? out_n + (size_t)r0 * g.H : nullptr;
            const int rc = grouped_layer(*layers[l], cur, mg, dst, dn, ws, ws_bytes, w, timeout_ns, st);
            if (rc) return rc;
            cur = dst;
        }
    }
    return MOE_OK;
}

}  // namespace moe
