// Internal declarations of libmoe_w4: workspace layout, kernel parameter
// blocks and the host-side launchers of each kernel family.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moe_w4.h"

namespace mw4 {

// Launch with programmatic dependent launch allowed when `pdl` is set: the
// kernel may be scheduled while the previous kernel on the stream finishes, so
// it must call griddep_wait() before it touches any memory (every kernel
// launched this way does so first; without the attribute that wait returns at
// once).  A refused attribute falls back to a plain launch.
template <typename... P, typename... A>
cudaError_t launch_pdl(bool pdl, void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const A&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess && pdl) {
        cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kern, args...);
    }
    return e;
}

constexpr int kGroup = 64;        // weights per scale/bias group
constexpr int kChunk = 128;       // tokens per grouping chunk
constexpr int kBM = 128;          // weight rows per tensor-core tile
constexpr int kBN = 128;          // token rows per tensor-core tile
constexpr int kBK = 64;           // reduction columns per pipeline stage (= one group)
constexpr int kDecodeMaxT = 16;   // largest decode batch
// Calls of at most this many rows chain their kernels with programmatic
// dependent launch (measured on H=2048, E=256, top-8, I=512: 8 rows 85.9 ->
// 81.8 us per call; a 4096-row chunk 0.386 -> 0.396 ms, so larger calls launch
// plainly).
constexpr int kPdlMaxT = 16;
inline bool pdl_for(int T) { return T <= kPdlMaxT; }
constexpr int kDecodeFusedRows = 5;   // default: decode calls of up to 5 rows run row by row (fused kernel)
constexpr int kRouterRowsPerCta = 256;  // H rows per decode-router CTA
constexpr int kRouterSplit = 2;         // prefill router: partial score arrays (halves of H)
// Width of one weight code: 4 (also for code_bits = 0) or 8.
inline int code_bits_of(const moe_w4_layer& L) { return L.code_bits == 8 ? 8 : 4; }
// FP8 E4M3 codes (one byte each, read as floats) instead of unsigned integers.
inline bool codes_e4m3(const moe_w4_layer& L) { return L.code_format == MOE_W4_CODES_E4M3; }

// Down projection: one CTA dequantises a 128-row weight tile once and runs it
// against up to this many 128-row blocks of the same expert, when its whole K
// (I columns) fits the tensor-memory A ring (kDownReuseMaxI columns).
constexpr int kDownBlocksPerUnit = 4;
// Word of the control header's pad[] holding the fused T=1 decode's call
// counter (the tag of its exchanged values is the counter + 1); kept across
// calls.
constexpr int kCtrlEpochWord = 61;
// Word of pad[] that the failure-detection test hook sets (0 in normal use):
// while it is non-zero, the T=1 kernel's CTA 0 does not publish its router
// scores, so every routed CTA's bounded wait for them runs out.
constexpr int kCtrlInjectWord = 60;
constexpr int kDownReuseMaxI = 512;
inline int down_blocks_per_unit(int I) { return I <= kDownReuseMaxI ? kDownBlocksPerUnit : 1; }
// Smallest token block the grouping may use (a tile override); sizes the block records.
constexpr int kMinBN = 32;

// Prefill tile choice: token rows per block (the GEMMs' N, at most kBN) and
// row blocks per down unit.  The default is kBN, and down_blocks_per_unit(I)
// once the routed rows average at least half a block per expert (T*k >= 64*E),
// else 1 (measured on GB300 at H=2048, I=512, E=256, top-8: units of 4 blocks
// 2% slower at T=512, 3-4% faster at T=2048 and 4096).  The environment
// variable MOE_W4_FORCE_TILE ("bn=64,du=2", either key optional) or
// moe_w4_set_tile_override replaces it, for ablations.
struct TileCfg { int bn, du; };
TileCfg tile_cfg(const moe_w4_layer& L, int T);

struct Ctrl;   // workspace control header (common.cuh)

// Records trace event `i` on `st` when tracing is enabled (moe_w4_set_trace_events).
void trace_mark(cudaStream_t st, int i);
// Records how many kernels the current traced call launches.
void trace_kernels(int n);

// Byte offsets of every region of the workspace (all 256-byte aligned).
struct WsLayout {
    size_t ctrl, logits, router_a, x16, topk_idx, topk_w, gamma, chunk_base, counts, offsets, perm, inv;
    size_t blkinfo, unitinfo, ntiles, hh, ys;
    size_t dec_part, dec_idx, dec_w, dec_gamma, dec_hh, dec_scores, dec_hx, dec_hsx;
    size_t total;
    int T_max, nchunk_max, max_blocks, max_tiles_gu, max_tiles_dn;
};
WsLayout ws_layout(const moe_w4_layer& L, int T_max);

// ---------------------------------------------------------------------------
// routing (router.cu, grouping.cu)
// ---------------------------------------------------------------------------
struct RouteOut {
    int32_t* topk_idx; float* topk_w; float* gamma;
    int32_t* counts;   // [E] routed (tile maps also need the shared group)
    int32_t* offsets;  // [E+1]
    int32_t* perm; int32_t* inv;
    int32_t* chunk_base;   // [chunks][E] assignments per (chunk of kChunk tokens, expert), counted by top-k
    float* logits;       // [kRouterSplit][T][E] partial router scores (tensor-core path), [T][E] otherwise
    uint16_t* router_a;  // [Epad][3H] bf16 split router weights, written per call unless the layer has them
    uint16_t* x16;     // fp16 copy of x written by the top-k kernel (NULL: not needed)
    int4* blkinfo; int32_t* ntiles;   // per-block records [max blocks] and tile counts [2]; NULL: no tile maps
    int4* unitinfo;                   // down units [max blocks]: {first block, blocks, group, 0}
    unsigned int* status;
};
cudaError_t launch_router_prefill(const moe_w4_layer& L, int T, const uint16_t* x, const RouteOut& o,
                                  cudaStream_t st);
// Bytes of the split router weights ([Epad][3H] bf16) and their one-time preparation.
size_t router_prep_bytes(const moe_w4_layer& L);
cudaError_t launch_router_prep(const moe_w4_layer& L, uint16_t* dst, cudaStream_t st);
// `force` (optional) replaces the tile choice (an ablation needs one-block down units).
cudaError_t launch_grouping(const moe_w4_layer& L, int T, const RouteOut& o, cudaStream_t st,
                            const TileCfg* force = nullptr);
// The grouping step on the host (ablation.cu): synchronises the stream, copies
// the top-k indices back, writes the same records as launch_grouping; sets
// *bad_index (and writes nothing) if an index is out of range.
cudaError_t host_grouping(const moe_w4_layer& L, int T, const RouteOut& o, cudaStream_t st, bool* bad_index);

// ---------------------------------------------------------------------------
// decode (decode.cu)
// ---------------------------------------------------------------------------
struct DecodeWs {
    float* part;        // [H/256][T][E] partial scores
    int32_t* idx;       // [T][k]
    float* w;           // [T][k]
    float* gamma;       // [T]
    float* hh;          // [T][k+1][I]
    unsigned int* counter;
    unsigned int* status;
    Ctrl* ctrl;         // control header (call counter of the fused kernel)
    uint64_t* fused_scores; // tagged partial router scores, fused_scores_bytes (fused T=1 kernel)
    uint64_t* fused_hx;     // tagged h of every slot, fp16 pairs, fused_hx_bytes (fused T=1 kernel)
    uint64_t* fused_hsx;    // tagged sums of 16-value pieces of h, fused_hsx_bytes (fused T=1 kernel)
};
bool decode_fused_supported(const moe_w4_layer& L);
// T rows as T consecutive cooperative launches of the fused batch-1 kernel
// (row t's routing at d.idx + t*k, d.w + t*k, d.gamma + t); returns the rows
// launched, fewer than T only when a launch was refused (nothing enqueued for
// the rest; the caller takes another path).
int launch_decode_fused_rows(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out, const DecodeWs& d,
                             cudaStream_t st);
// Decode calls of at most this many rows run row by row through the fused
// kernel when it covers the layer (moe_w4_set_decode_fused_rows overrides it).
int decode_fused_rows_max();
// Bytes of the fused kernel's exchange buffers for a layer: router score
// partials (replicated), h, and the sums of h's 32-value pieces.
size_t fused_scores_bytes(const moe_w4_layer& L);
size_t fused_hx_bytes(const moe_w4_layer& L);
size_t fused_hsx_bytes(const moe_w4_layer& L);
// The allocation-free decode: row by row through the fused kernel when it
// covers the layer, else (or when its first launch is refused) the three
// CUDA-core kernels of decode.cu.
cudaError_t launch_decode(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out, const DecodeWs& d,
                          cudaStream_t st);

// ---------------------------------------------------------------------------
// grouped tensor-core GEMMs (grouped_gemm.cu)
// ---------------------------------------------------------------------------
struct PrefillWs {
    const int4* blkinfo;     // per 128-row block of the grouped rows: {group (E = shared), first row, rows, first position}
    const int4* unitinfo;    // down units: {first row block, row blocks, group, 0}
    const int32_t* ntiles;   // [2] gate/up and down tile counts
    const int32_t* offsets; const int32_t* perm; const int32_t* inv;
    const float* topk_w; const float* gamma;
    const uint16_t* x16;  // fp16 [T][H]
    uint16_t* hh;   // fp16 [T*k + T][I]
    uint16_t* ys;   // fp16 [T*k + T][H]
    uint16_t* xg;   // fp16 [T*k][H]: token rows in grouped order, the gate/up B operand; shares ys's
                    // memory (read by gate/up only, before down writes ys)
    int max_tiles_gu, max_tiles_dn;
    unsigned int* status;
};
cudaError_t launch_grouped_ffn(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out,
                               const PrefillWs& p, cudaStream_t st,
                               const uint16_t* const* w16 = nullptr);
// The measurement-only separate dequantisation pass (ablation.cu): every weight
// of the layer's six matrices rebuilt in fp16, in the K order of the fused
// dequantisers, into w16 (moe_w4_ablation_scratch_bytes); w16_ptrs receives the
// six matrices' starts (gate, up, down, shared gate, shared up, shared down).
size_t f16_weights_bytes(const moe_w4_layer& L);
cudaError_t launch_f16_weights(const moe_w4_layer& L, uint16_t* w16, const uint16_t* w16_ptrs[6], unsigned int* status,
                               cudaStream_t st);

}  // namespace mw4
