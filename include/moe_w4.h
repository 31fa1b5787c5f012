/*
 * moe_w4.h -- C ABI of the GB300 (sm_103a) W4 group-affine sparse-MoE layer.
 *
 * One sparse mixture-of-experts feed-forward layer over 4-bit weights, as
 * described in "Optimizing on-device inference for Apple Silicon"
 * (perplexity.ai blog):
 *   - section "Qwen creates three different workload shapes": the router
 *     scores E = 256 experts per token and keeps the top k = 8; one shared
 *     expert processes every token;
 *   - section "Dequantise weights during matrix multiplication": each weight
 *     is a 4-bit code q; every group of 64 weights shares one bf16 scale s and
 *     one bf16 bias b, w = s*q + b; weights are rebuilt only at the point of
 *     use, products accumulate in fp32 and the output is bf16;
 *   - section "Keep expert routing on the GPU": histogram of assignments per
 *     expert, prefix scan to offsets, scatter of rows into expert groups and
 *     a block map, all without a CPU round trip;
 *   - sections "Optimise the single-row weight path" and "Reduce intermediate
 *     state and traffic": batch-1 decode is a fused GEMV (gate and up
 *     projections with the gated activation; output projection with the
 *     routing scores and the shared expert's result).
 * Readings taken where the pages are silent (also used by the oracle):
 *   routing weights = softmax over the k selected scores; equal scores pick
 *   the lower expert index; the shared expert is scaled by sigmoid(x . g);
 *   expert FFN = SwiGLU, y = Wd (silu(Wg x) * (Wu x)); rows of an expert
 *   group are ordered by ascending token index.
 *
 * Conventions for every entry point
 *   - All pointers except `L` itself are DEVICE pointers (the layer struct and
 *     its dims live in host memory).  The caller owns every buffer; the library
 *     never allocates, frees or synchronises.  All work is enqueued on
 *     `stream` (a cudaStream_t; 0 = legacy default stream) and returns at once.
 *   - bf16 values are passed as their 16-bit patterns (moe_w4_bf16).
 *   - Return 0 on success or a negative MOE_W4_ERR_* code; on error nothing
 *     has been enqueued, except MOE_W4_ERR_LAUNCH (a launch failed part-way;
 *     outputs are undefined).  No exception or abort crosses the ABI.
 *   - Results are deterministic: identical inputs give identical bytes, and
 *     rows are independent (a batch split into chunks gives the same rows).
 *   - Device-side faults of a bad pointer surface at the caller's next sync.
 */
#ifndef MOE_W4_H
#define MOE_W4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_w4_bf16; /* IEEE bfloat16 bit pattern */

/* One group-affine 4-bit matrix with `rows` output features and `cols` input
 * features (cols % 64 == 0):
 *   codes  uint32 [rows][cols/8]   eight 4-bit codes per word; input column
 *                                  8*w + i is nibble i of word w (nibble 0 =
 *                                  bits 0..3)
 *   scales bf16   [rows][cols/64]  scale of input columns 64g .. 64g+63
 *   biases bf16   [rows][cols/64]
 * Routed experts stack E such matrices contiguously (leading [E] axis). */
typedef struct {
    const uint32_t*    codes;
    const moe_w4_bf16* scales;
    const moe_w4_bf16* biases;
} moe_w4_mat;

/* The layer.  H hidden size, E routed experts, I intermediate size (routed and
 * shared), top_k experts kept per token, code_bits the width of one code.
 * Supported: H % 128 == 0, I % 128 == 0, 128 <= H <= 4096, 128 <= I <= 4096,
 * 1 <= E <= 1024, 1 <= top_k <= min(E, 8), code_bits 4 (or 0, read as 4) or 8.
 * Every pointer 16-byte aligned.
 * Codes: code_bits = 4: eight per uint32, the lowest column in the lowest
 * nibble (rows of cols/8 words); code_bits = 8: four per uint32, the lowest
 * column in the lowest byte (rows of cols/4 words).  Either way a weight is
 * s * q + b with q the unsigned code and s, b the bf16 scale and bias of its
 * group of 64 columns.  8-bit layers (either code_format below) take the
 * one-kernel batch-1 decode only for H = 2048, I = 512, E = 256, top_k = 8
 * (the grouped tensor-core path otherwise, and for decode calls of more rows
 * than moe_w4_set_decode_fused_rows); moe_w4_forward_decode_noalloc takes
 * them only where that one-kernel path applies (that shape, any T) and
 * returns MOE_W4_ERR_UNSUPPORTED otherwise.
 * code_format selects how a code is read (MOE_W4_CODES_*): unsigned integer
 * codes as above, or FP8 E4M3 codes (code_bits must be 8; same byte layout),
 * where a weight is s * v(q) + b with v(q) the E4M3 value of the byte: sign
 * bit 7, exponent field bits 6..3 with bias 7 (field 0: subnormal, m/8 * 2^-6),
 * mantissa field bits 2..0, no infinities, exponent and mantissa fields all
 * ones = NaN.  The format variant follows the "FP8 E4M3 decode, two codes per
 * half2" change listed in "To be verified: lithos-metal adds Apple inference
 * kernels" (aidaily), section "What was merged within one minute"; the E4M3
 * encoding is the one of "FP8 Formats for Deep Learning" (2022).  NaN codes
 * are not checked: they give NaN outputs. */
typedef struct {
    int H, E, I, top_k;
    const float* router_w;     /* [H][E] fp32                                   */
    const float* router_bias;  /* [E] fp32 added to the scores, or NULL         */
    const float* shared_gate;  /* [H] fp32; shared expert scale sigmoid(x . g)  */
    moe_w4_mat gate, up;       /* routed: [E][I][H/8] codes, [E][I][H/64] s, b  */
    moe_w4_mat down;           /* routed: [E][H][I/8] codes, [E][H][I/64] s, b  */
    moe_w4_mat sh_gate, sh_up; /* shared: [I][H/8] codes, [I][H/64] s, b        */
    moe_w4_mat sh_down;        /* shared: [H][I/8] codes, [H][I/64] s, b        */
    int code_bits;             /* 4 (or 0) or 8; with 8 the codes arrays hold
                                  cols/4 words per row instead of cols/8          */
    int code_format;           /* MOE_W4_CODES_UINT (0) or MOE_W4_CODES_E4M3    */
    const void* router_prep;   /* the router weights as moe_w4_prepare_router
                                  writes them (moe_w4_router_prep_bytes bytes,
                                  16-byte aligned), or NULL: the routing of
                                  every call on the grouped path then prepares
                                  them in its workspace first.  Must be rewritten after
                                  router_w changes.                            */
} moe_w4_layer;

enum {
    MOE_W4_CODES_UINT = 0,     /* unsigned integer codes, w = s * q + b         */
    MOE_W4_CODES_E4M3 = 1      /* FP8 E4M3 codes, w = s * v(q) + b; 8-bit only  */
};

enum {
    MOE_W4_OK              = 0,
    MOE_W4_ERR_INVALID     = -1, /* NULL pointer, T < 0, top_k out of range    */
    MOE_W4_ERR_UNSUPPORTED = -2, /* shape outside the supported set            */
    MOE_W4_ERR_WORKSPACE   = -3, /* workspace NULL, too small or misaligned    */
    MOE_W4_ERR_LAUNCH      = -4, /* a CUDA launch failed (cudaGetLastError)    */
    MOE_W4_ERR_DEVICE      = -5, /* reported by moe_w4_device_status: a kernel
                                    gave up a bounded wait or saw a bad index  */
    MOE_W4_ERR_ALIGN       = -6, /* a pointer is not 16-byte aligned           */
    MOE_W4_ERR_SCRATCH     = -7  /* moe_w4_forward_decode_noalloc: the call
                                    needs more than the fixed scratch array    */
};

/* The router weights prepared once per layer for the tensor-core scores of
 * the routing (prefill, and decode calls on the grouped path): W_r (fp32 [H][E]) split
 * exactly into three bf16 terms per weight, hi + mid + lo, stored transposed,
 * [ceil(E/128)*128][3H] bf16, rows past E zero.  The scores are unchanged by
 * the preparation; it only saves the split on every call.
 * moe_w4_router_prep_bytes: the size (0 if the layer is invalid).
 * moe_w4_prepare_router: writes them to `dst` (device memory owned by the
 * caller, dst_bytes >= that size, 16-byte aligned) on `stream`; reads only
 * L->router_w, L->H and L->E.  Returns MOE_W4_ERR_INVALID / _ALIGN /
 * _WORKSPACE (dst too small) or MOE_W4_ERR_LAUNCH.  Store dst in
 * L->router_prep to use it. */
size_t moe_w4_router_prep_bytes(const moe_w4_layer* L);
int moe_w4_prepare_router(const moe_w4_layer* L, void* dst, size_t dst_bytes, cudaStream_t stream);

/* Largest token count of one routing or prefill call (longer prompts are
 * chunked by the caller, as the benchmark's 4096-row chunks are): the kernels
 * index the T * (top_k + 1) grouped rows with 32-bit integers and tile the
 * tokens over at most 65535 router CTAs.  Larger T returns
 * MOE_W4_ERR_UNSUPPORTED (moe_w4_workspace_size: 0). */
#define MOE_W4_MAX_TOKENS (1 << 22)

/* Bytes of workspace needed for calls with up to T_max tokens (0 if the layer
 * is invalid or T_max is outside 0..MOE_W4_MAX_TOKENS).  The workspace holds
 * routing intermediates, the grouped activations and a small control header at
 * offset 0. */
size_t moe_w4_workspace_size(const moe_w4_layer* L, int T_max);

/* Clears the whole workspace (status word, completion counters, exchange
 * buffers).  Call once after allocating a workspace, before its first use, and
 * again after a call reported a device-side error; every later call leaves the
 * control header as it found it, except the sticky status word and a call
 * counter of the T=1 decode. */
int moe_w4_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Offset in bytes, within the workspace, of the int32 device status word:
 * 0 = no device-side error; otherwise a bit set of MOE_W4_STATUS_* values.
 * Kernels only OR into it; clear it with moe_w4_workspace_init. */
size_t moe_w4_status_offset(void);
#define MOE_W4_STATUS_WAIT_TIMEOUT 1u  /* a bounded wait gave up              */
#define MOE_W4_STATUS_BAD_INDEX    2u  /* a routing index was out of range    */
#define MOE_W4_STATUS_FP16_RANGE   4u  /* a value held in fp16 left its range
                                          (|v| > 65504): output not valid */
/* Value ranges.  The tensor-core paths hold activations (x), the weighted
 * SwiGLU output h, each expert's weighted output and the rebuilt weights
 * s * q + b (prefill and decode on the grouped path) in fp16; the one-kernel
 * batch-1 decode (also used row by row for small decode calls) holds x and h
 * in fp16 (with 4-bit codes half of their entries divided by 16, so x should
 * stay above about 1e-3 in magnitude for full precision there) and applies s
 * and b in fp32.  Inputs must therefore keep these within
 * the fp16 range: |x| <= 65504; per group |s| * qmax + |b| <= 65504 (qmax = 15
 * for 4-bit codes, 255 for 8-bit codes, 448 for E4M3); h and the expert outputs
 * <= 65504 in magnitude.  A kernel that sees a value beyond this sets
 * MOE_W4_STATUS_FP16_RANGE.  Below the fp16 normal range (6.1e-5) values keep
 * an absolute precision of 2^-25 rather than 11 significant bits: layers whose
 * rebuilt weights, h or expert outputs are mostly below it (scales around 1e-6
 * with unit activations) lose accuracy without any status bit.  Scale and
 * activation together: scales of 1e3 with activations of 1e-6 are in range. */

/* Routing of T tokens, 0 <= T <= MOE_W4_MAX_TOKENS (sections "Qwen creates three different workload
 * shapes" and "Keep expert routing on the GPU").
 *   x         bf16  [T][H]
 *   topk_idx  int32 [T][top_k]  selected experts, by descending score
 *   topk_w    fp32  [T][top_k]  softmax over the selected scores
 *   shared_gamma fp32 [T]       sigmoid(x . shared_gate)
 *   counts    int32 [E]         assignments per expert
 *   offsets   int32 [E+1]       exclusive prefix sum of counts
 *   perm      int32 [T*top_k]   perm[p] = t*top_k + j of the assignment at
 *                               grouped position p (tokens ascending in a group)
 *   inv       int32 [T*top_k]   inverse of perm
 * Scores are fp32 sums of x . W_r (+bias). */
int moe_w4_route(const moe_w4_layer* L, int T, const moe_w4_bf16* x,
                 int32_t* topk_idx, float* topk_w, float* shared_gamma,
                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                 void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Layer output for a decode batch, 1 <= T <= 16 (section "Optimise the
 * single-row weight path").  One row: one cooperative kernel for the whole
 * layer (router, W4 GEMVs for gate/up + SwiGLU and for down weighted by the
 * routing scores, plus the gated shared expert); its CTAs exchange router
 * scores and h through the workspace with bounded waits.  Up to
 * moe_w4_set_decode_fused_rows rows (5 by default): that kernel once per row,
 * in row order.  More rows, a shape that kernel does not cover, or a device
 * that refuses its cooperative launch: the grouped path of
 * moe_w4_forward_prefill, which reads each selected expert once for all rows
 * that chose it (moe_w4_decode_path tells which path a call takes).  out bf16
 * [T][H].  The one-kernel path reads the weights, router and shared gate
 * before it waits for the kernel that precedes it on the stream (programmatic
 * dependent launch): they must not be written by that kernel. */
int moe_w4_forward_decode(const moe_w4_layer* L, int T, const moe_w4_bf16* x,
                          moe_w4_bf16* out, void* workspace, size_t ws_bytes,
                          cudaStream_t stream);

/* The path moe_w4_forward_decode takes for T rows of layer L, into *path:
 * MOE_W4_PATH_FUSED_ROWS (the one-kernel batch-1 decode, once per row) or
 * MOE_W4_PATH_GROUPED (routing, grouping and grouped GEMMs; a refused
 * cooperative launch also ends there).  Host query on the current device.
 * Returns MOE_W4_ERR_INVALID (invalid layer, NULL path, T < 1),
 * MOE_W4_ERR_UNSUPPORTED (T > 16) or the layer checks' codes. */
#define MOE_W4_PATH_FUSED_ROWS 1
#define MOE_W4_PATH_GROUPED    2
int moe_w4_decode_path(const moe_w4_layer* L, int T, int* path);

/* Largest decode call (rows) that runs row by row through the one-kernel
 * batch-1 path, 1..16; 0 restores the default, 5 (measured on H=2048, E=256,
 * top-8, I=512: about 12.3 us per row back to back; the grouped path takes
 * 56, 61, 62 and 69 us at 2, 4, 5 and 6 rows).  1 keeps only single rows
 * there.
 * Process-wide; takes effect for calls enqueued afterwards.  Returns
 * MOE_W4_ERR_INVALID outside 0..16. */
int moe_w4_set_decode_fused_rows(int max_rows);

/* Layer output for a prefill batch, 1 <= T <= MOE_W4_MAX_TOKENS (section "Dequantise weights
 * during matrix multiplication"): routing as moe_w4_route, then grouped W4
 * GEMMs on the tensor cores (dequantised fp16 weight tiles and fp32
 * accumulators in tensor memory, fp16 activations) with a SwiGLU epilogue that
 * also applies the routing weight (or the shared gate), and an un-permute that
 * adds each token's k weighted expert outputs and the gated shared expert.
 * out bf16 [T][H].  The activations x, the weighted SwiGLU output and each
 * expert's weighted output must stay within the fp16 range (|v| <= 65504);
 * otherwise the status word gets MOE_W4_STATUS_FP16_RANGE. */
int moe_w4_forward_prefill(const moe_w4_layer* L, int T, const moe_w4_bf16* x,
                           moe_w4_bf16* out, void* workspace, size_t ws_bytes,
                           cudaStream_t stream);

/* Decode without any allocation, for callers that cannot allocate device
 * memory where they run the layer (an engine plugin whose host owns all
 * device memory, a real-time loop that must not wait on an allocator, a
 * memory plan fixed before the layer's shape is known).  The pages have no
 * counterpart: it is a deployment convenience of this library.
 * Same arguments as moe_w4_forward_decode, minus the workspace.  Where the
 * one-kernel batch-1 path covers the layer it runs that kernel once per row,
 * for every T (the grouped path's buffers would not fit); elsewhere, or when
 * its cooperative launch is refused, per-row CUDA-core GEMVs (router, gate/up,
 * down kernels; 4-bit codes only: a refused launch with one-byte codes returns
 * MOE_W4_ERR_LAUNCH), with results within the same tolerance of the oracle.  The
 * scratch lives in one fixed device array of
 * MOE_W4_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library keeps until the process exits.
 *   - Calls needing more scratch than that (large H, E or I, or many tokens)
 *     return MOE_W4_ERR_SCRATCH; the shapes used here (H=2048, E=256, I=512,
 *     top-8) fit for every T <= 16.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call reuses the same array and clears its control header first
 *     (except the one-kernel path's call counter);
 *     calls that overlap on the GPU (other streams, other threads) race and
 *     give wrong results: serialise them.
 *   - It never calls cudaMalloc, cudaFree or any allocating routine. */
#define MOE_W4_NOALLOC_SCRATCH_BYTES (2u << 20)
int moe_w4_forward_decode_noalloc(const moe_w4_layer* L, int T, const moe_w4_bf16* x,
                                  moe_w4_bf16* out, cudaStream_t stream);

/* Device status of the allocation-free decode: enqueues on `stream` a copy of
 * the status word inside the fixed scratch array (the MOE_W4_STATUS_* bits of
 * the allocation-free calls since the last one, as each call clears it first)
 * into *status, device or host memory; read it once the stream has passed this
 * point.  A non-zero word means the last call's output is not valid.  No
 * counterpart in the pages.  MOE_W4_ERR_INVALID for a NULL pointer,
 * MOE_W4_ERR_LAUNCH if the copy cannot be enqueued. */
int moe_w4_noalloc_status(unsigned int* status, cudaStream_t stream);

/* Failure-detection test hook for moe_w4_forward_decode_noalloc (no
 * production use; process-wide).  on != 0: in the following calls every
 * launch of the one-kernel batch-1 path (one per row) has one CTA skip
 * publishing its router scores, so the other CTAs'
 * bounded waits run out (after about 2 s): the call completes, its output is
 * not valid, and the status word (moe_w4_noalloc_status) gets
 * MOE_W4_STATUS_WAIT_TIMEOUT.  The aborting CTAs advance the call counter, so
 * the next call is valid.  No GPU fault, trap or hang is involved.  on = 0
 * turns it off.  Always returns MOE_W4_OK. */
int moe_w4_noalloc_test_skip_publish(int on);

/* Optional tracing for benchmarks: while set, every forward call records
 * events[0..n_events) (cudaEvent_t, created by the caller) on its stream:
 * event 0 before its first kernel and event i after its i-th kernel, so
 * consecutive events bracket one kernel each (prefill: 7 kernels -- router
 * scores, top-k, grouping, row gather, grouped gate/up GEMM, grouped down
 * GEMM, combine; decode on the grouped path: the same 7; decode row by row:
 * one fused kernel per row; three-kernel decode: router, gate/up GEMV, down
 * GEMV).  Extra kernels beyond n_events-1 are not traced; a call that
 * launches fewer kernels records its remaining events right after its last
 * kernel.  Events are recorded with
 * cudaEventRecordExternal, so they also fire inside a captured CUDA graph.
 * Pass NULL to stop tracing.  Process-wide setting, not thread-safe. */
int moe_w4_set_trace_events(cudaEvent_t* events, int n_events);

/* Prefill tile override, for ablations ("Optimizing on-device inference for
 * Apple Silicon", section "Match tile size to expert load": the tile height is
 * chosen per workload).  bn: token rows per block of the grouped GEMMs (the
 * MMA's N), 32, 64 or 128 (the default); du: row blocks of one expert that a
 * down-projection weight tile is dequantised once for, 1, 2 or 4 (by default 4
 * where I <= 512 and T * top_k >= 64 * E, else 1; with I > 512 du > 1 is
 * ignored).  0 restores a default.  The environment variable MOE_W4_FORCE_TILE ("bn=64,du=2", either
 * key optional) is read once, at the first prefill call or at the first call
 * of this function, which then replaces it.  Process-wide; takes effect for
 * calls enqueued afterwards.  Returns MOE_W4_ERR_INVALID for other values. */
int moe_w4_set_tile_override(int bn, int du);

/* Failure-detection test hook (no production use).  on != 0: the next batch-1
 * decode calls on this workspace have one CTA skip publishing its router
 * scores, so the other CTAs' bounded waits for them run out (after about 2 s):
 * the call completes, its output is not valid, and the status word gets
 * MOE_W4_STATUS_WAIT_TIMEOUT.  No GPU fault, trap or hang is involved.  on = 0
 * (or moe_w4_workspace_init, which must follow any device-side error anyway)
 * turns it off. */
int moe_w4_test_skip_publish(void* workspace, size_t ws_bytes, int on, cudaStream_t stream);

/* Failure-detection test hook (no production use; process-wide): rows >= 0
 * makes every following decode call (moe_w4_forward_decode and
 * moe_w4_forward_decode_noalloc) launch the one-kernel batch-1 path for at
 * most `rows` of its rows and then take the fallback it takes when a
 * cooperative launch is refused: the grouped path for the remaining rows (the
 * per-row CUDA-core kernels in the allocation-free decode, or
 * MOE_W4_ERR_LAUNCH there for one-byte codes).  Nothing is launched and
 * refused for real.  rows < 0 turns it off.  Always returns MOE_W4_OK. */
int moe_w4_test_refuse_fused_after(int rows);

/* Test hook: the block records of the last prefill (or grouped-path decode) call
 * enqueued on `workspace` for T tokens, copied on `stream` to `dst` (device
 * memory, at least moe_w4_test_block_records_bytes(L, T) bytes): two int32
 * tile counts (gate/up blocks x I/128, down units x H/128), then one record of
 * four int32 per block of grouped rows: expert (E for the shared expert's
 * group), first row within the expert's group, rows, first grouped position.
 * Blocks are listed expert by expert, routed experts first; only the first
 * (tile count 0) / (I/128) records are meaningful.  ("Optimizing on-device
 * inference for Apple Silicon", section "Keep expert routing on the GPU": the
 * list of fixed-size blocks the grouped product processes.)  Returns
 * MOE_W4_ERR_INVALID / _WORKSPACE or MOE_W4_ERR_LAUNCH. */
size_t moe_w4_test_block_records_bytes(const moe_w4_layer* L, int T);
int moe_w4_test_block_records(const moe_w4_layer* L, int T, const void* workspace, size_t ws_bytes,
                              int32_t* dst, size_t dst_bytes, cudaStream_t stream);

/* Number of kernels the most recent traced call launched (0 before any). */
int moe_w4_last_traced_kernels(void);

/* Static description of a status code. */
const char* moe_w4_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4_H */
