// Internal definitions shared by the host ABI (moe_abi.cu), the packer
// (moe_pack.cu) and the decode kernel (moe_layer.cu).  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

constexpr int kGroup = 64;          // affine group along the contraction axis
constexpr int kSub = 16;            // codes per sub-group (one lane step)
constexpr int kMaxRows = 8;         // token rows per launch (larger M is chunked)
constexpr int kMaxLayers = 64;      // layers per persistent launch
constexpr int kMaxStages = 64;      // ring stages (mbarrier pairs)
constexpr int kMaxE = 512;
constexpr int kMaxK = 32;
constexpr int kMaxGPL = 4;          // 64-groups per lane of a row: K <= 32 * 64 * kMaxGPL
constexpr int kLogitCopies = 8;     // copies of the router logits in the workspace (readers spread over them)
constexpr int kMaxCtas = 160;       // CTAs of a persistent launch (one per SM) at most
constexpr int kRouterRowsCta = 4;   // router rows one CTA reduces and publishes, at most
constexpr int kActCopies = 1;       // copies of the exchanged activations (more copies measured slower)
constexpr int kCtrlBytes = 2048;    // control block at the start of the workspace
constexpr int kSmemMax = 232448;    // dynamic shared memory per CTA on sm_100-class parts

// Status word bits (workspace control block).
constexpr int kStatusTimeout = 1;
constexpr int kStatusBounds = 2;
constexpr int kStatusNotResident = 4;   // a selected expert had no cache slot (streamed layers)

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bytes of one packed row of K inputs: LSB-first code stream, then one
// 32-bit word (scale | bias << 16) per 64-group, padded to 16 bytes.
// bits == 0: K fp32 values.
__host__ __device__ constexpr int row_bytes(int K, int bits)
{
    return bits == 0 ? (int)align_up((size_t)K * 4, 16)
                     : (int)align_up((size_t)K * bits / 8 + (size_t)(K / kGroup) * 4, 16);
}

// Input-major copy of the router (the persistent kernel's partial logits:
// each CTA dots every router row with its own slice of the input, so it
// reads a range of input columns of all rows).  Er rows padded to Erp, a
// multiple of 16.  Quantised routers: one code byte per (column, row),
// [H][Erp], then one word (scale | bias << 16) per (group, row), [H/64][Erp].
// fp32 routers: [H][Erp] floats.
__host__ __device__ constexpr size_t router_t_bytes(int H, int Erp, int bits)
{
    return bits == 0 ? (size_t)H * Erp * 4 : (size_t)H * Erp + (size_t)(H / kGroup) * Erp * 4;
}

// Bytes of a CTA's slice of that copy: nh columns of every row and the
// scale/bias words of the ng groups they touch (multiples of 16 bytes).
__host__ __device__ constexpr int router_slice_bytes(int nh, int ng, int Erp, int bits)
{
    return bits == 0 ? nh * Erp * 4 : nh * Erp + ng * Erp * 4;
}

// Geometry of a layer: sizes, row sizes, blob offsets, launch plan.
struct Geo {
    int H, I, E, k, Is;
    int has_shared, rb, sb, qb;     // routed / shared / router bits
    int Er;                         // router rows = E + has_shared (last = shared gate)
    int Erp;                        // Er rounded up to 16 (rows of the input-major router copy)
    int rr_bytes;                   // router row
    int g_bytes;                    // routed gate (or up) row, K = H
    int d_bytes;                    // routed down row, K = I
    int sg_bytes;                   // shared gate (or up) row, K = H
    int sd_bytes;                   // shared down row, K = Is
    float eps;
    // blob offsets (bytes)
    size_t off_router, off_gamma, off_gamma_next, off_router_t, off_gu, off_down, off_sgu, off_sdown, total;
    size_t rt_sb;                   // scale/bias words inside the input-major router copy (H * Erp)
};

// Per-layer device pointers inside the packed blob.
struct LayerPtrs {
    const uint8_t *router;
    const uint8_t *router_t; // input-major router copy (router_t_bytes)
    const uint8_t *gu;       // E * I units of (gate row, up row)
    const uint8_t *down;     // E * H rows
    const uint8_t *sgu;      // I_shared units
    const uint8_t *sdown;    // H rows
    const uint16_t *gamma;
    const uint16_t *gamma_next;  // NULL when absent
    // Streamed layers (moe_streamed_*): the routed experts live in host
    // memory and gu / down are an HBM cache of n_slots experts; slot_of[e]
    // is expert e's slot (or -1).  NULL for a resident layer.
    const int32_t *slot_of;
    int n_slots;
};

// Workspace layout (offsets from the workspace base).
struct WsLayout {
    int maxr;                // rows per launch
    int max_slots;           // distinct routed experts per launch
    size_t off_logits, off_act, off_act_s, off_ping, off_part, off_stage_in, off_stage_out, total;
    size_t act_cs, act_s_cs; // words of one copy of the routed / shared activations
    int max_M;               // rows the host-staging area holds
    // Grouped mode (M above maxr: the tensor-core expert path), sized for
    // grp_rows = min(max_M, kGroupRows) rows and grp_slots = min(E, grp_rows k)
    // distinct experts; all zero when max_M <= maxr.
    int grp_rows, grp_slots;
    size_t off_g_hn, off_g_sigma, off_g_idx, off_g_w, off_g_slotof, off_g_experts, off_g_masks, off_g_count;
    size_t off_g_act, off_g_act_s, off_g_y, off_g_ysh, off_g_ping;
};

constexpr int kGroupRows = 32;      // token rows of one grouped pass (mask width)

struct Ctrl {                // first kCtrlBytes of the workspace
    unsigned count;          // unused (kept zero)
    unsigned pad0[31];
    unsigned exit;           // CTAs of the running launch that have finished (own 128-byte line)
    unsigned pad1[31];
    int status;              // kStatus* bits
    int where;               // debug: which wait gave up
    int pad2[30];
    unsigned seq;            // launches completed on this workspace (mod kSeqWrap): the tag range
    unsigned pad3[31];       // of a launch is seq * 64 + 1 .. seq * 64 + 64
};
// seq wraps before seq * 64 + 64 passes 2^32; the launch that wraps clears
// every tagged word of the workspace first, so no earlier word can match.
constexpr unsigned kSeqWrap = 1u << 26;
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

// Launch plan of the persistent kernel.
struct Plan {
    int P;                   // CTAs (one per SM)
    int S;                   // stage bytes
    int NS;                  // ring stages
    int maxr;                // rows per launch
    int max_slots;
    int hrows;               // output rows per CTA (upper bound, even)
    int pb_bytes;            // prefetch buffer (gamma, the CTA's router slice, shared units of a layer)
    int act_pairs;           // (slot, row) activation vectors the staging buffer holds
    int smem_bytes;
    int ncw;                 // compute warps of the kernel build the plan is for
};

enum Mode { kModeLayers = 0, kModeRouter = 1 };

struct KParams {
    Geo g;
    Plan p;
    int L;                   // layers in this launch
    LayerPtrs layer[kMaxLayers];
    const uint16_t *x;       // [M, H] input of the first layer
    int M;
    uint16_t *out;           // [M, H] output of the last layer
    uint16_t *out_normed;    // [M, H] or NULL
    int32_t *idx_out;        // router mode
    float *w_out;            // router mode
    int mode;
    uint8_t *ws;             // workspace base
    WsLayout ws_l;
    long long timeout_ns;
    int skip_row;            // debug: router logit row left unpublished in layer 0 (-1 = none)
    int inject_e;            // checked build only: id row 0 of layer 0 reports as its first choice (-1 = none)
    unsigned long long *trace;   // optional per-CTA phase timestamps (ns), NULL = off
};

constexpr int kTraceEvents = 24; // events recorded per (CTA, layer)

bool make_geo(const moe_layer_desc &d, Geo &g);
void make_ws_layout(const Geo &g, int max_M, WsLayout &w);
// The decode kernel is built for two numbers of compute warps (each CTA has
// one more, the producer): 11 for launches of at most 4 token rows of at
// most 2048 inputs, where more warps hide more of the row kernels' latency,
// and 8 otherwise: wider rows' gate/up units would be cut into twice as
// many ring stages (bulk copies), and with more rows the staging buffer
// leaves the 22-stage ring too little room (8 rows: 351 against 190 us per
// layer).  Registers are given to warps in fours, so both builds get 168
// per thread.  make_plan / launch_decode are the 11-warp build, the _w8
// entries the 8-warp one; decode_plan / decode_launch pick.
inline int decode_warps(const Geo &g, int maxr) { return g.H <= 2048 && maxr <= 4 ? 11 : 8; }
bool make_plan(const Geo &g, int maxr, int num_sms, Plan &p);
bool make_plan_w8(const Geo &g, int maxr, int num_sms, Plan &p);
inline bool decode_plan(const Geo &g, int maxr, int num_sms, Plan &p)
{
    return decode_warps(g, maxr) == 8 ? make_plan_w8(g, maxr, num_sms, p) : make_plan(g, maxr, num_sms, p);
}
int rows_per_launch(int H);
int device_sms();

}  // namespace moe

struct moe_layer {
    moe_layer_desc desc;
    moe::Geo geo;
    uint8_t *base;
    size_t bytes;
    moe::LayerPtrs ptrs;
};

struct moe_stack {
    int L;
    moe_layer **layers;
};

struct moe_qkv {
    moe_qkv_desc desc;
    int rows;          // n_q + n_k + n_v
    int row_bytes;
    uint8_t *base;     // packed rows (borrowed)
};

// Host-side entry points of the kernels (moe_layer.cu, moe_pack.cu, moe_tc.cu,
// moe_grouped.cu).
namespace moe {
int launch_decode(const KParams &kp, cudaStream_t stream);
int launch_decode_w8(const KParams &kp, cudaStream_t stream);
inline int decode_launch(const KParams &kp, cudaStream_t stream)
{
    return kp.p.ncw == 8 ? launch_decode_w8(kp, stream) : launch_decode(kp, stream);
}
int launch_pack(const moe_layer &L, const moe_src_layer &src, cudaStream_t stream);
// rows of one matrix into consecutive packed rows at dst (moe_pack.cu)
int launch_pack_rows(const moe_src_matrix &m, int bits, int rows, int K, uint8_t *dst, cudaStream_t stream);
// fused Q/K/V projection (moe_layer.cu)
int launch_qkv(const uint8_t *W, int rows, int K, int bits, const uint16_t *x, int M, float *y, int *err,
               long long timeout_ns, cudaStream_t stream);
// split-K decode attention with grouped query heads (moe_attn.cu)
size_t attn_workspace_bytes(int T_cap);
int attn_max_positions();
int launch_attn(const uint16_t *q, const uint16_t *k, const uint16_t *vt, int T_cap, int pos0, int M, float *o,
                void *ws, int *err, long long timeout_ns, cudaStream_t stream);
int launch_attn_append(const uint16_t *kn, const uint16_t *vn, int M, int pos0, uint16_t *kc, uint16_t *vtc, int T_cap,
                       cudaStream_t stream);
int launch_export(const moe_layer &L, int tensor_id, int expert, uint8_t *codes, uint16_t *scales,
                  uint16_t *biases, cudaStream_t stream);
// One set of grouped tensor-core products (moe_tc.cu): slot u's expert
// experts[u], rows of masks[u]; W rows e * rows .., K inputs, row_bytes per
// packed row; inputs in[(u * in_u + m) * K ..]; U_dev a device-side slot
// count or NULL.
struct TcSetHost {
    const uint8_t *W;
    int rows, K, row_bytes;
    const float *in;
    int in_u;
    const int32_t *experts;
    const uint32_t *masks;
    const int *U_dev;
    float *out;
};
int launch_grouped_tc2(bool swiglu, int bits_a, const TcSetHost &a, int nA, int bits_b, const TcSetHost *b, int nB,
                       int M, int *err, long long timeout_ns, cudaStream_t stream);
int launch_grouped_fma(bool swiglu, int bits_a, const TcSetHost &a, int nA, int bits_b, const TcSetHost *b, int nB,
                       int M, int *err, long long timeout_ns, cudaStream_t stream);
int launch_grouped_tc(int bits, bool swiglu, const uint8_t *W, int rows, int K, int row_bytes, const float *in, int in_u,
                      int M, const int32_t *experts, const uint32_t *masks, int U, const int *U_dev, float *out,
                      int *err, long long timeout_ns, cudaStream_t stream);
int launch_gate_up_tc(const moe_layer &L, const float *hn, int M, const int32_t *experts, const uint32_t *masks, int U,
                      float *act, int *err, long long timeout_ns, cudaStream_t stream);
int launch_down_tc(const moe_layer &L, const float *act, int M, const int32_t *experts, const uint32_t *masks, int U,
                   float *y, int *err, long long timeout_ns, cudaStream_t stream);
int grouped_forward(const moe_layer *const *layers, int L, const uint16_t *x, int M, uint16_t *out, uint16_t *out_n,
                    void *ws_dev, size_t ws_bytes, long long timeout_ns, cudaStream_t st);
void note_cuda_error(int err);
void note_launch();
bool grouped_products_tc();   // moe_set_grouped_products
}  // namespace moe
