/*
 * moe.h -- C ABI of the GB300 (sm_103a) quantized MoE decode-layer library.
 *
 * The layer is the decode step of a top-k mixture-of-experts FFN over affine
 * group-quantised expert weights, as described by:
 *   - PureDrive-35B-A3B-MLX model card (huggingface.co), "Summary": 256
 *     experts, top-8 plus a shared expert, 6-bit experts, 8-bit shared
 *     weights; "How it works": a verify pass of 1 + draft rows reads the
 *     weights once and every row is identical to a one-row decode; fused
 *     add + RMSNorm;
 *   - flash-moe (ja.news.hada.io topic 27758), "FMA最適化デクォントカーネル":
 *     dequantised weight = code * scale + bias; "Metal Compute Shaders":
 *     dequant mat-vec, SwiGLU, RMS normalisation, MoE combine + residual +
 *     gate; "Deferred GPU Expert Compute": combine, norm and residual stay on
 *     the GPU and feed the next layer.
 *
 * Per token row m (rows never interact):
 *   hn      = x_m / sqrt(mean(x_m^2) + eps) * gamma
 *   logits  = W_r hn ;  p = softmax(logits) ;  top-k of p (ties: lower id),
 *             w_i = p_i / sum_topk p
 *   y_e     = W_d,e (silu(W_g,e hn) * (W_u,e hn))           (each selected e)
 *   sigma   = sigmoid(w_sg . hn) ; y_s = shared-expert FFN of hn
 *   out_m   = bf16(x_m + sum_i w_i y_i + sigma y_s)
 *   outn_m  = bf16(out_m / sqrt(mean(out_m^2) + eps) * gamma_next)
 * Every matrix is stored as groups of 64 consecutive elements along its input
 * (contraction) axis, w = q * s + b with a b-bit code q and bf16 s, b.
 *
 * Conventions for every call:
 *   - Return value: a moe_status.  No call throws, aborts or exits.
 *   - Memory: the library never allocates device memory.  The caller owns
 *     every device buffer (weights, workspace, inputs, outputs) and keeps it
 *     alive while a handle or an enqueued call uses it.  Handles are small
 *     host structs (malloc) that borrow those device pointers.
 *   - Pointers named *_dev are device pointers; everything else is host.
 *     bf16 values travel as uint16_t bit patterns.
 *   - Streams: calls taking a stream only enqueue work on it and return;
 *     errors raised while the kernels run are read with moe_stream_status().
 *   - Sizes: H, I, I_shared multiples of 64 (H >= 256), E <= 512, k <= min(E, 32),
 *     routed/shared bits in {4, 6, 8}, router bits in {0 (fp32), 8}.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,      /* NULL pointer, negative size, inconsistent descriptors */
    MOE_ERR_UNSUPPORTED = 2,      /* sizes or bit widths outside the supported set */
    MOE_ERR_BUFFER_TOO_SMALL = 3, /* weight blob or workspace smaller than the *_size query */
    MOE_ERR_CUDA = 4,             /* a CUDA runtime call failed; see moe_last_cuda_error() */
    MOE_ERR_TIMEOUT = 5,          /* a device-side wait gave up (the kernel returned early) */
    MOE_ERR_DEVICE = 6,           /* a device-side check failed (bounds build) */
    MOE_ERR_NOT_RESIDENT = 7      /* a streamed layer's selected expert was not in its cache */
} moe_status;

/* Shape and storage of one layer. */
typedef struct moe_layer_desc {
    int H;            /* hidden size */
    int I;            /* routed expert intermediate size */
    int E;            /* routed experts */
    int k;            /* experts kept per row */
    int routed_bits;  /* 4, 6 or 8 */
    int shared_bits;  /* 4, 6 or 8 (ignored when has_shared == 0) */
    int router_bits;  /* 0 = fp32 router rows, 8 = 8-bit groups; also used for the shared-gate vector */
    int has_shared;   /* 1 = a sigmoid-gated shared expert is present */
    int I_shared;     /* shared expert intermediate size (has_shared == 1) */
    float eps;        /* RMSNorm epsilon */
} moe_layer_desc;

/* One source matrix [rows, cols] in canonical form, device pointers:
 * either codes (uint8, one code per byte, row-major) + scales + biases (bf16,
 * [rows, cols/64]), or fp32 weights w (row-major) which the packer quantises:
 *   s = bf16((max - min) / (2^b - 1)), b = bf16(min),
 *   q = clamp(rint((w - b) / s), 0, 2^b - 1)  (fp32 arithmetic, q = 0 when s == 0).
 * A router with router_bits == 0 must be given as fp32 w and stays fp32. */
typedef struct moe_src_matrix {
    const uint8_t *codes_dev;
    const uint16_t *scales_dev;
    const uint16_t *biases_dev;
    const float *w_dev;
} moe_src_matrix;

/* All source tensors of one layer (device pointers). */
typedef struct moe_src_layer {
    moe_src_matrix gate;         /* [E * I, H]: expert e rows e*I .. e*I + I - 1 */
    moe_src_matrix up;           /* [E * I, H] */
    moe_src_matrix down;         /* [E * H, I] */
    moe_src_matrix shared_gate;  /* [I_shared, H] */
    moe_src_matrix shared_up;    /* [I_shared, H] */
    moe_src_matrix shared_down;  /* [H, I_shared] */
    moe_src_matrix router;       /* [E, H] */
    moe_src_matrix sgate;        /* [1, H] shared-expert gate vector */
    const uint16_t *gamma_dev;       /* [H] RMSNorm weight of this layer's input */
    const uint16_t *gamma_next_dev;  /* [H] RMSNorm weight applied to the output, or NULL */
} moe_src_layer;

typedef struct moe_layer moe_layer;
typedef struct moe_stack moe_stack;

/* Tensor ids for moe_export_canonical. */
enum {
    MOE_T_ROUTER = 0, MOE_T_SGATE = 1, MOE_T_GATE = 2, MOE_T_UP = 3, MOE_T_DOWN = 4,
    MOE_T_SHARED_GATE = 5, MOE_T_SHARED_UP = 6, MOE_T_SHARED_DOWN = 7
};

/* Bytes of the packed device blob of one layer (codes as LSB-first bit
 * streams, per-group bf16 scale and bias, rows padded to 16 bytes; the
 * router also input-major, one code byte per weight, so that the decode
 * kernel's CTAs can each fetch a column slice of every router row).
 * Errors: MOE_ERR_INVALID_ARG (NULL), MOE_ERR_UNSUPPORTED (sizes/bits). */
int moe_pack_size(const moe_layer_desc *desc, size_t *weight_bytes);

/* Affine group quantisation / packing into the device layout (flash-moe,
 * "FMA最適化デクォントカーネル": w = code * scale + bias; group 64 along the
 * input axis).  Reads the canonical sources in `src`, writes the blob at
 * dst_dev (dst_bytes >= moe_pack_size), enqueued on `stream`, and returns a
 * handle in *out that borrows dst_dev.  The sources may be freed once the
 * stream has passed this call.
 * Errors: INVALID_ARG, UNSUPPORTED, BUFFER_TOO_SMALL, CUDA. */
int moe_pack_weights(const moe_layer_desc *desc, const moe_src_layer *src, void *dst_dev,
                     size_t dst_bytes, moe_layer **out, moe_stream_t stream);

/* Frees the handle (not the blob).  NULL is a no-op. */
void moe_layer_destroy(moe_layer *layer);

/* Writes one quantised matrix of a packed layer back in canonical form
 * (codes one per byte, bf16 scales and biases) to device buffers sized like
 * the moe_src_matrix of that tensor; `expert` selects the routed expert for
 * MOE_T_GATE/UP/DOWN.  Errors: INVALID_ARG, UNSUPPORTED (fp32 router), CUDA. */
int moe_export_canonical(const moe_layer *layer, int tensor_id, int expert, uint8_t *codes_dev,
                         uint16_t *scales_dev, uint16_t *biases_dev, moe_stream_t stream);

/* Scratch bytes needed by the decode calls for up to max_M rows per call
 * (partial router dots, logits, expert activations, inter-layer activations
 * and a control block).
 * The same workspace serves every call on one stream; calls that run at the
 * same time on the GPU need separate workspaces. */
int moe_workspace_size(const moe_layer_desc *desc, int max_M, size_t *ws_bytes);

/* Zeroes the workspace: the control block (launch counter, status word)
 * and every word the kernels exchange.  Call once after allocating a
 * workspace, and again after any call reported MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE. */
int moe_workspace_init(void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Router only (RMSNorm, router mat-vec, softmax, top-k, renormalisation) for
 * M rows of x_dev [M, H] bf16.  Writes idx_dev [M, k] int32 (descending
 * weight, ties to the lower expert id) and w_dev [M, k] fp32 (sums to 1 per
 * row).  PureDrive model card, "Summary": the full top-8 of 256 is kept.
 * Errors: INVALID_ARG, UNSUPPORTED (M < 1 or M > max_M of the workspace),
 * BUFFER_TOO_SMALL, CUDA. */
int moe_router_topk(const moe_layer *layer, const uint16_t *x_dev, int M, int32_t *idx_dev,
                    float *w_dev, void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* One layer for M rows of x_dev [M, H] bf16: writes out_dev [M, H] (bf16
 * residual stream) and, when out_normed_dev != NULL, the fused next RMSNorm
 * out_normed_dev [M, H] (needs gamma_next).  out_dev may alias x_dev.  Each
 * selected expert's weights are streamed from memory once for all the rows
 * that chose it (model card, "How it works": the verify pass reads its
 * weights once).  Up to one persistent launch's rows (8 at H = 2048) row m
 * of the result is bitwise the one-row result; above, grouped mode runs
 * (moe_set_grouped): the same routing, values within the tolerance.
 * Errors: INVALID_ARG, UNSUPPORTED, BUFFER_TOO_SMALL, CUDA. */
int moe_decode_layer(const moe_layer *layer, const uint16_t *x_dev, int M, uint16_t *out_dev,
                     uint16_t *out_normed_dev, void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* A stack of L layers with identical descriptors: x_{l+1} = out_l.  The
 * handle borrows the layer handles.  flash-moe, "Deferred GPU Expert
 * Compute": combine, norm and residual stay on the GPU and feed the next
 * layer; here the whole stack runs in one persistent launch (per 64 layers
 * and per chunk of rows) with no host round trip between layers.
 * Errors: INVALID_ARG (NULL, L < 1, descriptors differ). */
int moe_stack_create(moe_layer *const *layers, int L, moe_stack **out);

/* Runs the stack on x_dev [M, H]; writes the last layer's out_dev [M, H] and,
 * when out_normed_dev != NULL, its fused next RMSNorm.  out_dev may alias x_dev.
 * Errors: as moe_decode_layer. */
int moe_stack_forward(moe_stack *stack, const uint16_t *x_dev, int M, uint16_t *out_dev,
                      uint16_t *out_normed_dev, void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* moe_stack_forward from host buffers: copies x_host [M, H] to the device
 * (into the workspace, which must be sized for M rows), runs the stack,
 * copies out_host [M, H] back and synchronises the stream.  Pinned host
 * memory gives the fastest copies.  Returns the stream status. */
int moe_stack_forward_host(moe_stack *stack, const uint16_t *x_host, int M, uint16_t *out_host,
                           void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Frees the stack handle (not the layers).  NULL is a no-op. */
void moe_stack_destroy(moe_stack *stack);

/* moe_decode_layer without a caller-provided workspace, for callers that
 * cannot allocate device memory at the point of the call: code enqueued
 * while a stream is being captured into a CUDA graph (cudaMalloc is not
 * allowed there), plug-ins that run inside another framework's memory pool
 * and may not grow it, and latency-critical paths that must not take an
 * allocation's implicit synchronisation.  The pages describing the method
 * have no counterpart of this call; it exists for such callers only.
 *
 * The scratch lives in a fixed array of MOE_NOALLOC_SCRATCH_BYTES of device
 * memory inside the library (every GPU that loads the library holds it
 * until the process exits).  The call always runs the persistent kernel in
 * launches of one launch's rows (8 at H = 2048) and never grouped mode,
 * whatever moe_set_grouped says; its bound is therefore that kernel's part
 * of the workspace layout (moe_workspace_size without the grouped-mode
 * regions, which only calls of more rows than one launch include).  Calls
 * whose persistent-kernel layout exceeds the array are rejected with
 * MOE_ERR_BUFFER_TOO_SMALL before anything is enqueued; so is every other
 * argument error: a rejected call enqueues nothing.  Inputs and outputs are
 * as for moe_decode_layer.
 *
 * - The first call on a device looks up the array's device address on that
 *   device (once, cudaGetSymbolAddress); make that first call outside any
 *   stream capture.  The address is cached per device for the life of the
 *   process; after cudaDeviceReset it is stale and the call must not be used.
 * - Each accepted call clears the array's control block (status word,
 *   barrier counters) on `stream` before its kernels, so an earlier failed
 *   call does not affect it; the status word therefore describes the most
 *   recent call only: read it with moe_noalloc_status before the next call.
 * - Every call on a device shares the one array: calls that can overlap on
 *   the GPU (different streams without ordering between them) race and give
 *   wrong results.  Order them on one stream.
 * - No device memory is allocated or freed by this call.
 * Errors: INVALID_ARG, UNSUPPORTED (shape, or a device index above 63),
 * BUFFER_TOO_SMALL (scratch too small), CUDA; errors raised while the
 * kernels run (a device wait that gave up) are read with moe_noalloc_status. */
#define MOE_NOALLOC_SCRATCH_BYTES (16u << 20)
int moe_decode_layer_noalloc(const moe_layer *layer, const uint16_t *x_dev, int M, uint16_t *out_dev,
                             uint16_t *out_normed_dev, moe_stream_t stream);

/* Synchronises `stream` and returns the status of the latest
 * moe_decode_layer_noalloc call on the current device: MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE from the scratch array's status word
 * (or MOE_ERR_CUDA).  The paper has no counterpart of this call either. */
int moe_noalloc_status(moe_stream_t stream);

/* Synchronises `stream` and returns MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE
 * from the workspace status word (or MOE_ERR_CUDA). */
int moe_stream_status(void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Test hook: the next decode calls leave router logit `skip_row` (an expert
 * index; -1 = off) of their first layer unpublished, so that every CTA's
 * wait for it runs out, and give every device wait `timeout_ns` (<= 0
 * restores the default of 2 s).  Used to check that a wait that runs out
 * returns MOE_ERR_TIMEOUT instead of hanging. */
int moe_debug_set(int skip_row, long long timeout_ns);

/* Build flags of the loaded library: MOE_BUILD_DEBUG_BOUNDS is set in the
 * bounds-checked build (libmoe_debug.so, compiled with MOE_DEBUG_BOUNDS).
 * In that build the persistent kernel compares every index it computes from
 * data (the expert ids out of the top-k, slot and activation-pair numbers)
 * with the size of the array it indexes before the access; an index out of
 * range sets a bit of the workspace status word, is replaced by 0 so that
 * the launch stays inside its buffers and runs to its end, and the call (or
 * moe_stream_status) returns MOE_ERR_DEVICE.  The checked build computes the
 * same results as the normal one when no check fails.  No CUDA call; never
 * fails. */
#define MOE_BUILD_DEBUG_BOUNDS 1
int moe_build_flags(void);

/* Test hook of the bounds-checked build: while expert >= 0, the next decode
 * calls on the persistent kernel make token row 0 of their first layer
 * report `expert` as its first routing choice, as a faulty top-k would;
 * an id >= E is caught by the checks above (MOE_ERR_DEVICE).  expert < 0
 * turns it off.  Host state only.  Returns MOE_ERR_UNSUPPORTED in the
 * normal build, which has neither the hook nor the checks. */
int moe_debug_inject(int expert);

/* Diagnostic hook: while set, every decode launch records globaltimer
 * stamps (ns) into trace_dev: [CTA][layer][24] as uint64 for the first
 * min(layers, 64) layers of a launch, followed by a per-warp timeline of two
 * CTAs, [2][64][16][16]; bytes must cover (SMs * 64 * 24 + 2 * 64 * 256) * 8.
 * NULL turns it off.  The stamps show where the time of
 * each layer goes (per phase, per CTA). */
int moe_debug_trace(void *trace_dev, size_t bytes);

/* Grouped mode for many rows.  moe_decode_layer and moe_stack_forward run
 * calls of more rows than one persistent launch holds (M > 8 at H = 2048),
 * and of at least min_rows rows, in groups of up to 32 rows per layer:
 * RMSNorm and fp32 router logits, the warp top-k per row (bit-exact routing
 * wherever the top-k logit gap exceeds fp32 rounding), every selected
 * expert read once for the group's rows with its products on the tensor
 * cores (the arithmetic of moe_gate_up_tc and moe_down_tc), then the
 * combine with the residual and the fused next RMSNorm.  Values are within
 * the one-row path's tolerance but not bitwise equal to it.  The default,
 * min_rows = 1, takes grouped mode whenever M exceeds one launch; min_rows = 0
 * keeps every M on the FMA path (launches of 8 rows, each re-reading the
 * experts its rows share), where every row of any M is bitwise its one-row
 * result: a row-exact verify caller with more rows than one launch sets
 * min_rows = 0.  The grouped regions of the workspace are included in
 * moe_workspace_size whenever max_M exceeds one launch.  Process-wide;
 * returns INVALID_ARG for min_rows < 0. */
int moe_set_grouped(int min_rows);

/* Grouped mode's expert products: 0 (the default) on the FMA pipes, each
 * selected expert's rows read once and dotted with each of its token rows
 * by the persistent kernel's one-vector row kernel (about 1.7 token rows per
 * expert at 32 rows with top-8 of 256 experts, where the tensor-core tiles
 * would be mostly padding); 1 on the tensor cores (the products of
 * moe_gate_up_tc and moe_down_tc).  Widths above 2048 always use the tensor
 * cores.  Process-wide; INVALID_ARG for other values. */
int moe_set_grouped_products(int tensor_cores);

/* Grouped gate/up of routed experts on the tensor cores (tcgen05 MMAs,
 * fp32 accumulators in tensor memory): the first half of each selected
 * expert's FFN for every token row that chose it, when many rows share an
 * expert (flash-moe, "Metal Compute Shaders": dequant mat-vec and SwiGLU;
 * PureDrive-35B-A3B model card, "How it works": one read of the weights for
 * all rows).  Grouped mode (moe_set_grouped) computes a layer's expert
 * products with these kernels; this call exposes the gate/up half alone.
 *
 *   for u < U, e = experts_dev[u], each row m < M with bit m of masks_dev[u]:
 *     act_dev[(u * M + m) * I + j] = silu(W_gate,e[j] . hn_m) * (W_up,e[j] . hn_m)
 *
 * hn_dev: fp32 [M][H], rows already normalised (device).  experts_dev int32 [U]
 * and masks_dev uint32 [U] (device).  act_dev: fp32 [U][M][I] (device); entries
 * of rows outside a mask are not written (mask bits at or above M are
 * ignored).  M <= 32.  Arithmetic: each weight w = q * s + b (fp32) and each
 * input value v are split into two fp16 halves: hi is v with its 13 low
 * mantissa bits cleared (exact in fp16), lo = fp16(v - hi).  The four half
 * products accumulate in fp32, each chunk of 64 inputs in its own sum added
 * into fp32 registers, so every term keeps ~21 significant bits.  Inputs and
 * weights must stay below 65504 in magnitude.  err_dev (device int) is set to 1 if a device
 * wait runs out (see moe_debug_set); the caller clears it.
 * Errors: INVALID_ARG (NULL pointer, M < 1, U < 0), UNSUPPORTED (M > 32),
 * CUDA (launch failed). */
int moe_gate_up_tc(const moe_layer *layer, const float *hn_dev, int M, const int32_t *experts_dev,
                   const uint32_t *masks_dev, int U, float *act_dev, int *err_dev, moe_stream_t stream);

/* The down projection of the same experts on the tensor cores, same
 * arithmetic (flash-moe, "Metal Compute Shaders": dequant mat-vec of the
 * down matrix; the weighted combine is not part of this call):
 *
 *   y_dev[(u * M + m) * H + h] = W_down,e[h] . act_dev[(u * M + m) * I ..]
 *
 * for u < U, e = experts_dev[u], each row m of masks_dev[u].  act_dev fp32
 * [U][M][I] (moe_gate_up_tc's output), y_dev fp32 [U][M][H] (device); rows
 * outside a mask are not read or written.  Errors: as moe_gate_up_tc, and
 * UNSUPPORTED when H is not a multiple of 128. */
int moe_down_tc(const moe_layer *layer, const float *act_dev, int M, const int32_t *experts_dev,
                const uint32_t *masks_dev, int U, float *y_dev, int *err_dev, moe_stream_t stream);

/* ------------------------------------------------------------------ */
/* Fused Q/K/V projection.  "Qwen3.5-397B on M5 Max" (openclawradar),
 * 効果的な最適化: the attention's Q, K and V projections are fused so that
 * the input row is read once; the PureDrive-35B-A3B-MLX model card,
 * "Summary", keeps attention weights at 8 bits.  The input is the layer's
 * normalised activations, e.g. the out_normed rows a moe_decode_layer or
 * moe_stack_forward call writes:
 *
 *   y[m, r] = W[r] . x_m,  W = [W_q; W_k; W_v] stacked row-wise ([n, H], n =
 *   n_q + n_k + n_v), every row in affine groups of 64 along H (w = q * s + b,
 *   bf16 s and b), x bf16 [M, H], y fp32 [M, n]: Q in columns [0, n_q), K in
 *   [n_q, n_q + n_k), V after.
 *
 * The kernel streams each row block from memory once for all M rows; the
 * rows of y are bitwise independent of M. */
typedef struct moe_qkv_desc {
    int H;      /* input width (multiple of 64, >= 128) */
    int n_q;    /* rows of the Q projection (heads x head dim) */
    int n_k;    /* rows of the K projection */
    int n_v;    /* rows of the V projection */
    int bits;   /* 4, 6 or 8 */
} moe_qkv_desc;

typedef struct moe_qkv moe_qkv;

/* Bytes of the packed projection (rows of moe_pack_size's row format).
 * Errors: INVALID_ARG (NULL), UNSUPPORTED (sizes, bits). */
int moe_qkv_pack_size(const moe_qkv_desc *desc, size_t *bytes);

/* Packs the three matrices (each a moe_src_matrix of [n_x, H]: canonical
 * codes/scales/biases, or fp32 weights that are quantised as for the layer)
 * into dst_dev (>= moe_qkv_pack_size bytes, 256-byte aligned) on `stream`, and
 * returns a handle that borrows dst_dev.  Errors: INVALID_ARG, UNSUPPORTED,
 * BUFFER_TOO_SMALL, CUDA. */
int moe_qkv_pack(const moe_qkv_desc *desc, const moe_src_matrix *q, const moe_src_matrix *k,
                 const moe_src_matrix *v, void *dst_dev, size_t dst_bytes, moe_qkv **out, moe_stream_t stream);

/* y_dev[M, n] (fp32) = the projection of x_dev [M, H] (bf16, 16-byte
 * aligned), enqueued on `stream`.  err_dev (a device int the caller zeroes)
 * is set to 1 if a device wait runs out (see moe_debug_set).  M >= 1 and small
 * enough that the M input rows fit in shared memory (M * H <= 32768).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
int moe_qkv_forward(const moe_qkv *qkv, const uint16_t *x_dev, int M, float *y_dev, int *err_dev,
                    moe_stream_t stream);

/* Frees the handle (not the packed rows).  NULL is a no-op. */
void moe_qkv_destroy(moe_qkv *qkv);

/* ------------------------------------------------------------------------
 * Decode attention with grouped query heads, split over the keys
 * (PureDrive-35B-A3B-MLX model card, "How it works": one attention kernel
 * for the one-row decode and the multi-row verify, reading K/V once for all
 * query heads of a group and all verify rows, split flash-decoding style
 * with split points and summation order that depend only on the row's
 * position; "Beyond this checkpoint": 16 query heads, 2 KV heads, head
 * dimension 256).  The shape is fixed at those sizes.
 *
 * Cache layout (caller-owned device memory, bf16):
 *   k_cache  [2][T_cap][256]  key of position t of key/value head g at
 *            (g * T_cap + t) * 256;
 *   vt_cache [2][256][T_cap]  values stored transposed: value d of position t
 *            of head g at (g * 256 + d) * T_cap + t.
 * T_cap must be a multiple of 8, at most MOE_ATTN_MAX_POSITIONS, and both
 * base addresses 16-byte aligned.  Positions past the last valid one are
 * never used.
 *
 * moe_attn_workspace_size: device scratch a call with this T_cap needs
 * (the per-chunk partial results and the merge's per-segment sums and
 * counters; no initialisation needed).  Calls that can run at the same time
 * on the GPU need separate scratch.  Errors: INVALID_ARG. */
#define MOE_ATTN_Q_HEADS 16
#define MOE_ATTN_KV_HEADS 2
#define MOE_ATTN_HEAD_DIM 256
#define MOE_ATTN_MAX_ROWS 8
#define MOE_ATTN_MAX_POSITIONS (1 << 19)
int moe_attn_workspace_size(int T_cap, size_t *bytes);

/* Attention of M token rows (1 <= M <= 8) at positions pos0 .. pos0 + M - 1
 * against the cache, whose positions 0 .. pos0 + M - 1 hold valid keys and
 * values (the rows' own included, see moe_attn_append): row m attends to
 * positions 0 .. pos0 + m,
 *   o[m][h] = sum_t softmax_t(q[m][h] . k[g][t] / 16) v[g][t], g = h / 8.
 * q_dev bf16 [M][16][256]; o_dev fp32 [M][16][256].  The keys are split into
 * chunks of 512 positions, one CTA per (chunk, KV head) on the tensor cores
 * (scores and weighted values in fp32, the softmax weights as two bf16
 * halves), then a merge of each row's chunks in order: row m's result is
 * bitwise the same for any M.  err_dev (int, device) is set to 1 if a device
 * wait runs out of time; the caller clears it.  Two launches, asynchronous
 * on `stream`.  Errors: INVALID_ARG (null or misaligned pointers, M or pos0
 * out of range, T_cap not a multiple of 8), BUFFER_TOO_SMALL, UNSUPPORTED
 * (no tensor-map encoder in the driver), CUDA. */
int moe_attn_decode(const uint16_t *q_dev, const uint16_t *k_cache_dev, const uint16_t *vt_cache_dev, int T_cap,
                    int pos0, int M, float *o_dev, void *ws_dev, size_t ws_bytes, int *err_dev,
                    moe_stream_t stream);

/* Writes the keys and values of M new rows (bf16 [M][2][256] each) into the
 * cache at positions pos0 .. pos0 + M - 1 (values transposed).  One launch.
 * Errors: INVALID_ARG, CUDA. */
int moe_attn_append(const uint16_t *k_new_dev, const uint16_t *v_new_dev, int M, int pos0, uint16_t *k_cache_dev,
                    uint16_t *vt_cache_dev, int T_cap, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Streamed layers: the routed experts of a layer live in host memory (the
 * Grace side of a GB300, over NVLink-C2C) and only the experts the router
 * selects are copied into an HBM cache of n_slots expert slots, least
 * recently used evicted first (flash-moe, "SSD Expert Streaming" and
 * "Trust the OS": only the selected experts are loaded, an LRU cache keeps
 * the popular ones; AiiStream Q3.6 article: the next layer's experts are
 * predicted and loaded ahead; "Qwen3.5-397B on M5 Max": temporal expert
 * prediction).  The router, norm weights and shared expert stay in HBM.
 * A streamed layer decodes with the same kernel as a resident one and gives
 * the same bits; it runs on the persistent path only (never grouped mode,
 * and the tensor-core product calls refuse it).
 *
 * moe_streamed_size: device bytes of a streamed layer with n_slots slots
 * (k <= n_slots <= E): the resident parts, the cache and the slot map.
 * Errors: INVALID_ARG, UNSUPPORTED. */
typedef struct moe_streamed moe_streamed;
int moe_streamed_size(const moe_layer_desc *desc, int n_slots, size_t *dev_bytes);

/* Makes a streamed layer from a packed one: the whole blob is copied to
 * host_blob (host memory the caller allocated, pinned for asynchronous
 * copies, at least moe_pack_size bytes, kept alive by the caller), the
 * resident parts to dev_buf (256-byte aligned, moe_streamed_size bytes);
 * the cache starts empty.  Synchronises `stream`; afterwards the packed
 * layer and its device memory may be released.  Errors: INVALID_ARG,
 * BUFFER_TOO_SMALL, CUDA. */
int moe_streamed_create(const moe_layer *packed, void *host_blob, size_t host_bytes, void *dev_buf, size_t dev_bytes,
                        int n_slots, moe_streamed **out, moe_stream_t stream);

/* The layer handle to pass to moe_decode_layer / moe_router_topk /
 * moe_stack_create.  A decode whose routing selects an expert without a
 * cache slot reports MOE_ERR_NOT_RESIDENT (moe_stream_status) and its
 * output is not defined. */
const moe_layer *moe_streamed_layer(const moe_streamed *s);

/* Makes experts expert_ids[0 .. n) (host array, repeats allowed) resident:
 * the missing ones are copied from host memory on `stream` (two copies per
 * expert: its gate/up units and its down rows), evicting the least
 * recently used slots that hold none of the listed experts, then the slot
 * map is updated on `stream`.  *fetched (may be NULL) = experts copied.
 * Counts hits and misses.  Errors: INVALID_ARG (an id outside 0 .. E - 1),
 * BUFFER_TOO_SMALL (more distinct ids than slots), CUDA. */
int moe_streamed_prepare(moe_streamed *s, const int32_t *expert_ids, int n, moe_stream_t stream, int *fetched);

/* Counters since creation: hits and misses of moe_streamed_prepare and of
 * the routing in moe_streamed_forward, experts fetched and their bytes (also
 * by prefetches), experts predicted for this layer and how many of the
 * selected experts the prediction named.  Any pointer may be NULL. */
int moe_streamed_stats(const moe_streamed *s, long long *hits, long long *misses, long long *fetched,
                       long long *bytes, long long *predicted, long long *predicted_used);

void moe_streamed_destroy(moe_streamed *s);

/* One forward of M rows (M <= one persistent launch's rows) through L
 * streamed layers of one shape, in the library's runtime: for each layer,
 * route it on its input (moe_router_topk), wait for the routing on the
 * host, make its selected experts resident, decode it (out_dev; layer l > 0
 * reads and overwrites out_dev; the last layer also writes out_normed_dev
 * when given).  With predict != 0, layer l + 1's router also runs on layer
 * l's input, and the experts it names are copied into layer l + 1's cache
 * on copy_stream while layer l is decoded (the copy waits for the last
 * decode that read that cache; layer l + 1's decode waits for the copy).
 * Kernels run on `stream` only.  route_dev: device scratch of at least
 * 16 * M * k bytes.  Errors: as the calls above; UNSUPPORTED for M above
 * one launch. */
int moe_streamed_forward(moe_streamed *const *layers, int L, const uint16_t *x_dev, int M, uint16_t *out_dev,
                         uint16_t *out_normed_dev, void *ws_dev, size_t ws_bytes, void *route_dev, size_t route_bytes,
                         int predict, moe_stream_t stream, moe_stream_t copy_stream);

/* Human-readable name of a status code (static string). */
const char *moe_status_str(int status);

/* The last CUDA error code seen by the library on this host thread (0 = none). */
int moe_last_cuda_error(void);

/* Host-side checks (no GPU needed): the code-extraction tables the kernels
 * use; the launch plans of the test shapes against the invariants the
 * kernel relies on (ring depth, stage and buffer sizes, shared-memory limit);
 * and the workspace layouts for 1 to 100 rows (aligned, ordered regions, each
 * large enough for what is written into it, grouped-mode regions only above
 * one launch's rows).  Returns the number of violations, 0 when consistent. */
int moe_selftest_host(void);

/* Number of kernel launches the library enqueued on this host thread since
 * the last reset (reset = 1 zeroes it after reading). */
long long moe_launch_count(int reset);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
