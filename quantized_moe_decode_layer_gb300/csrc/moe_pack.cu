// Affine group quantisation and packing into the device layout, and the
// reverse export to canonical form.
//
// flash-moe (ja.news.hada.io topic 27758), "FMA最適化デクォントカーネル": the
// dequantised weight is code * scale + bias.  Groups are 64 consecutive
// elements along the input axis with a bf16 scale and bias each.
//
// Device row layout (row_bytes(K, bits) bytes, 16-byte multiple):
//   [K codes as one LSB-first bit stream: code i at bits i*b .. i*b+b-1]
//   [K/64 words: scale bf16 | bias bf16 << 16]
//   [zero padding]
// fp32 rows (router_bits == 0) are K floats.
#include <cuda_bf16.h>

#include "moe_internal.h"

namespace moe {
namespace {

struct PackSrc {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint16_t *biases;
    const float *w;
};

// Destination of source row r: base + r * stride + offset.
struct PackDst {
    uint8_t *base;
    size_t stride;
    size_t offset;
};

__device__ __forceinline__ uint16_t bf16_rn(float v)
{
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ float bf16_val(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Quantise one group of 64 fp32 values: s = bf16((max-min)/(2^b-1)),
// b = bf16(min), q = clamp(rint((w-b)/s)); fp32 arithmetic throughout.
template <int BITS>
__device__ void quantize64(const float *w, uint8_t *q, uint16_t &sb, uint16_t &bb)
{
    float mn = w[0], mx = w[0];
    for (int i = 1; i < 64; ++i) {
        float v = w[i];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    const int qmax = (1 << BITS) - 1;
    float range = __fsub_rn(mx, mn);
    float sf = __fdiv_rn(range, (float)qmax);
    sb = bf16_rn(sf);
    bb = bf16_rn(mn);
    float s = bf16_val(sb), b = bf16_val(bb);
    for (int i = 0; i < 64; ++i) {
        int code = 0;
        if (s != 0.0f) {
            float r = rintf(__fdiv_rn(__fsub_rn(w[i], b), s));
            r = r < 0.0f ? 0.0f : r;
            r = r > (float)qmax ? (float)qmax : r;
            code = (int)r;
        }
        q[i] = (uint8_t)code;
    }
}

template <int BITS>
__global__ void pack_kernel(PackSrc src, PackDst dst, int rows, int K)
{
    const int groups = K / kGroup;
    const long long total = (long long)rows * groups;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(t / groups), g = (int)(t % groups);
        uint8_t *row = dst.base + (size_t)r * dst.stride + dst.offset;
        if constexpr (BITS == 0) {
            const float4 *s4 = reinterpret_cast<const float4 *>(src.w + (size_t)r * K + (size_t)g * 64);
            float4 *d4 = reinterpret_cast<float4 *>(row + (size_t)g * 256);
            for (int i = 0; i < 16; ++i) d4[i] = s4[i];
        } else {
        uint8_t q[64];
        uint16_t sb, bb;
        if (src.codes) {
            const uint8_t *c = src.codes + (size_t)r * K + (size_t)g * 64;
            for (int i = 0; i < 64; ++i) q[i] = c[i] & ((1 << BITS) - 1);
            sb = src.scales[(size_t)r * groups + g];
            bb = src.biases[(size_t)r * groups + g];
        } else {
            float w[64];
            const float *s = src.w + (size_t)r * K + (size_t)g * 64;
            for (int i = 0; i < 64; ++i) w[i] = s[i];
            quantize64<BITS>(w, q, sb, bb);
        }
        constexpr int NW = 2 * BITS;  // 32-bit words per 64 codes
        uint32_t words[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) words[i] = 0;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const int o = i * BITS, wi = o >> 5, sh = o & 31;
            words[wi] |= (uint32_t)q[i] << sh;
            if (sh + BITS > 32) words[wi + 1] |= (uint32_t)q[i] >> (32 - sh);
        }
        uint32_t *dw = reinterpret_cast<uint32_t *>(row + (size_t)g * 8 * BITS);
#pragma unroll
        for (int i = 0; i < NW; ++i) dw[i] = words[i];
        uint32_t *sbw = reinterpret_cast<uint32_t *>(row + (size_t)K * BITS / 8);
        sbw[g] = (uint32_t)sb | ((uint32_t)bb << 16);
        }
    }
}

template <int BITS>
__global__ void export_kernel(const uint8_t *base, size_t stride, size_t offset, int rows, int K,
                              uint8_t *codes, uint16_t *scales, uint16_t *biases)
{
    const int groups = K / kGroup;
    const long long total = (long long)rows * groups;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(t / groups), g = (int)(t % groups);
        const uint8_t *row = base + (size_t)r * stride + offset;
        const uint32_t *dw = reinterpret_cast<const uint32_t *>(row + (size_t)g * 8 * BITS);
        for (int i = 0; i < 64; ++i) {
            const int o = i * BITS, wi = o >> 5, sh = o & 31;
            uint32_t v = dw[wi] >> sh;
            if (sh + BITS > 32) v |= dw[wi + 1] << (32 - sh);
            codes[(size_t)r * K + (size_t)g * 64 + i] = (uint8_t)(v & ((1u << BITS) - 1));
        }
        const uint32_t sbw = reinterpret_cast<const uint32_t *>(row + (size_t)K * BITS / 8)[g];
        scales[(size_t)r * groups + g] = (uint16_t)(sbw & 0xFFFF);
        biases[(size_t)r * groups + g] = (uint16_t)(sbw >> 16);
    }
}

// The input-major router copy (router_t_bytes) from the packed router rows:
// code (column h, row e) as one byte at h * Erp + e, and row e's scale/bias
// word of group g at H * Erp + g * Erp + e (fp32 routers: the value at
// h * Erp + e).  Consecutive threads take consecutive rows of one column.
// Rows Er .. Erp - 1 stay as the caller cleared them (zero).
template <int BITS>
__global__ void router_t_kernel(const uint8_t *rows, int rr_bytes, int Er, int H, int Erp, uint8_t *dst)
{
    const long long total = (long long)Er * H;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(t % Er), h = (int)(t / Er);
        const uint8_t *row = rows + (size_t)e * rr_bytes;
        if constexpr (BITS == 0) {
            reinterpret_cast<float *>(dst)[(size_t)h * Erp + e] = reinterpret_cast<const float *>(row)[h];
        } else {
            const uint32_t *dw = reinterpret_cast<const uint32_t *>(row);
            const int o = h * BITS, wi = o >> 5, sh = o & 31;
            uint32_t v = dw[wi] >> sh;
            if (sh + BITS > 32) v |= dw[wi + 1] << (32 - sh);
            dst[(size_t)h * Erp + e] = (uint8_t)(v & ((1u << BITS) - 1u));
            if ((h & (kGroup - 1)) == 0) {
                const uint32_t sbw = reinterpret_cast<const uint32_t *>(row + (size_t)H * BITS / 8)[h / kGroup];
                reinterpret_cast<uint32_t *>(dst + (size_t)H * Erp)[(size_t)(h / kGroup) * Erp + e] = sbw;
            }
        }
    }
}

int grid_for(long long work)
{
    long long b = (work + 255) / 256;
    return (int)(b < 1 ? 1 : (b > 4096 ? 4096 : b));
}

int router_t_fill(const Geo &g, uint8_t *b, cudaStream_t st)
{
    const int grid = grid_for((long long)g.Er * g.H);
    const uint8_t *rows = b + g.off_router;
    uint8_t *dst = b + g.off_router_t;
    switch (g.qb) {
    case 0: router_t_kernel<0><<<grid, 256, 0, st>>>(rows, g.rr_bytes, g.Er, g.H, g.Erp, dst); break;
    case 4: router_t_kernel<4><<<grid, 256, 0, st>>>(rows, g.rr_bytes, g.Er, g.H, g.Erp, dst); break;
    case 6: router_t_kernel<6><<<grid, 256, 0, st>>>(rows, g.rr_bytes, g.Er, g.H, g.Erp, dst); break;
    case 8: router_t_kernel<8><<<grid, 256, 0, st>>>(rows, g.rr_bytes, g.Er, g.H, g.Erp, dst); break;
    default: return MOE_ERR_UNSUPPORTED;
    }
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

int pack_matrix(const moe_src_matrix &m, int bits, int rows, int K, PackDst dst, cudaStream_t st)
{
    if (bits == 0 ? !m.w_dev : (!m.w_dev && (!m.codes_dev || !m.scales_dev || !m.biases_dev)))
        return MOE_ERR_INVALID_ARG;
    PackSrc s{m.codes_dev, m.scales_dev, m.biases_dev, m.w_dev};
    const long long work = (long long)rows * (K / kGroup);
    const int grid = grid_for(work);
    switch (bits) {
    case 0: pack_kernel<0><<<grid, 256, 0, st>>>(s, dst, rows, K); break;
    case 4: pack_kernel<4><<<grid, 256, 0, st>>>(s, dst, rows, K); break;
    case 6: pack_kernel<6><<<grid, 256, 0, st>>>(s, dst, rows, K); break;
    case 8: pack_kernel<8><<<grid, 256, 0, st>>>(s, dst, rows, K); break;
    default: return MOE_ERR_UNSUPPORTED;
    }
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

}  // namespace

int launch_pack_rows(const moe_src_matrix &m, int bits, int rows, int K, uint8_t *dst, cudaStream_t st)
{
    return pack_matrix(m, bits, rows, K, PackDst{dst, (size_t)row_bytes(K, bits), 0}, st);
}

int launch_pack(const moe_layer &L, const moe_src_layer &src, cudaStream_t st)
{
    const Geo &g = L.geo;
    uint8_t *b = L.base;
    cudaError_t e = cudaMemsetAsync(b, 0, g.total, st);
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    int rc;
    const size_t unit = 2 * (size_t)g.g_bytes;
    if ((rc = pack_matrix(src.gate, g.rb, g.E * g.I, g.H, PackDst{b + g.off_gu, unit, 0}, st))) return rc;
    if ((rc = pack_matrix(src.up, g.rb, g.E * g.I, g.H, PackDst{b + g.off_gu, unit, (size_t)g.g_bytes}, st))) return rc;
    if ((rc = pack_matrix(src.down, g.rb, g.E * g.H, g.I, PackDst{b + g.off_down, (size_t)g.d_bytes, 0}, st))) return rc;
    if ((rc = pack_matrix(src.router, g.qb, g.E, g.H, PackDst{b + g.off_router, (size_t)g.rr_bytes, 0}, st))) return rc;
    if (g.has_shared) {
        const size_t sunit = 2 * (size_t)g.sg_bytes;
        if ((rc = pack_matrix(src.shared_gate, g.sb, g.Is, g.H, PackDst{b + g.off_sgu, sunit, 0}, st))) return rc;
        if ((rc = pack_matrix(src.shared_up, g.sb, g.Is, g.H, PackDst{b + g.off_sgu, sunit, (size_t)g.sg_bytes}, st))) return rc;
        if ((rc = pack_matrix(src.shared_down, g.sb, g.H, g.Is, PackDst{b + g.off_sdown, (size_t)g.sd_bytes, 0}, st))) return rc;
        if ((rc = pack_matrix(src.sgate, g.qb, 1, g.H,
                              PackDst{b + g.off_router + (size_t)g.E * g.rr_bytes, (size_t)g.rr_bytes, 0}, st)))
            return rc;
    }
    if ((rc = router_t_fill(g, b, st))) return rc;
    e = cudaMemcpyAsync(b + g.off_gamma, src.gamma_dev, (size_t)g.H * 2, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && src.gamma_next_dev)
        e = cudaMemcpyAsync(b + g.off_gamma_next, src.gamma_next_dev, (size_t)g.H * 2, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

int launch_export(const moe_layer &L, int tensor_id, int expert, uint8_t *codes, uint16_t *scales,
                  uint16_t *biases, cudaStream_t st)
{
    const Geo &g = L.geo;
    const uint8_t *b = L.base;
    const uint8_t *base = nullptr;
    size_t stride = 0, offset = 0;
    int rows = 0, K = 0, bits = 0;
    const size_t unit = 2 * (size_t)g.g_bytes, sunit = 2 * (size_t)g.sg_bytes;
    switch (tensor_id) {
    case MOE_T_ROUTER: base = b + g.off_router; stride = g.rr_bytes; rows = g.E; K = g.H; bits = g.qb; break;
    case MOE_T_SGATE:
        base = b + g.off_router + (size_t)g.E * g.rr_bytes; stride = g.rr_bytes; rows = 1; K = g.H; bits = g.qb;
        if (!g.has_shared) return MOE_ERR_INVALID_ARG;
        break;
    case MOE_T_GATE: case MOE_T_UP:
        if (expert < 0 || expert >= g.E) return MOE_ERR_INVALID_ARG;
        base = b + g.off_gu + (size_t)expert * g.I * unit; stride = unit;
        offset = tensor_id == MOE_T_UP ? (size_t)g.g_bytes : 0; rows = g.I; K = g.H; bits = g.rb;
        break;
    case MOE_T_DOWN:
        if (expert < 0 || expert >= g.E) return MOE_ERR_INVALID_ARG;
        base = b + g.off_down + (size_t)expert * g.H * g.d_bytes; stride = g.d_bytes; rows = g.H; K = g.I; bits = g.rb;
        break;
    case MOE_T_SHARED_GATE: case MOE_T_SHARED_UP:
        if (!g.has_shared) return MOE_ERR_INVALID_ARG;
        base = b + g.off_sgu; stride = sunit; offset = tensor_id == MOE_T_SHARED_UP ? (size_t)g.sg_bytes : 0;
        rows = g.Is; K = g.H; bits = g.sb;
        break;
    case MOE_T_SHARED_DOWN:
        if (!g.has_shared) return MOE_ERR_INVALID_ARG;
        base = b + g.off_sdown; stride = g.sd_bytes; rows = g.H; K = g.Is; bits = g.sb;
        break;
    default: return MOE_ERR_INVALID_ARG;
    }
    const int grid = grid_for((long long)rows * (K / kGroup));
    switch (bits) {
    case 4: export_kernel<4><<<grid, 256, 0, st>>>(base, stride, offset, rows, K, codes, scales, biases); break;
    case 6: export_kernel<6><<<grid, 256, 0, st>>>(base, stride, offset, rows, K, codes, scales, biases); break;
    case 8: export_kernel<8><<<grid, 256, 0, st>>>(base, stride, offset, rows, K, codes, scales, biases); break;
    default: return MOE_ERR_UNSUPPORTED;
    }
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { note_cuda_error((int)e); return MOE_ERR_CUDA; }
    return MOE_OK;
}

}  // namespace moe
