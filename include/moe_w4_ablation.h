/* Measurement-only entry point of libmoe_w4: the prefill with one step of the
 * path replaced by the design the source pages measured against, so that the
 * gain of the product's design can be re-measured on this GPU.  Not for
 * production use.
 *
 * ("Optimizing on-device inference for Apple Silicon", section "Keep expert
 * routing on the GPU": a routing step synchronised with the CPU between the
 * router and the expert GEMMs, against the histogram, scan and scatter kept
 * on the GPU; section "Dequantise weights during matrix multiplication": a
 * separate pass that expands the 4-bit weights to a 16-bit array the matmul
 * then reads, against rebuilding each weight tile on chip.)
 */
#ifndef MOE_W4_ABLATION_H
#define MOE_W4_ABLATION_H

#include "moe_w4.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
    /* The router and top-k run on the GPU as usual; the stream is then
     * synchronised, the top-k indices copied to the host, the expert
     * histogram, scan, positions and block records computed there and copied
     * back before the grouped GEMMs are enqueued.  Same output as
     * moe_w4_forward_prefill (the records are identical).  The call blocks the
     * host until the routing is done and cannot be captured in a CUDA graph. */
    MOE_W4_ABLATE_HOST_ROUTING = 1,
    /* Every weight of the layer (all E routed experts and the shared one) is
     * first rebuilt in fp16 into `scratch` by a separate pass (the values and
     * K order the fused dequantisers produce), then the grouped GEMMs read
     * those fp16 tiles by TMA and multiply them from shared memory; down
     * units are one row block each.  Same output as moe_w4_forward_prefill,
     * bit for bit. */
    MOE_W4_ABLATE_SEPARATE_DEQUANT = 2
};

/* Bytes of `scratch` that moe_w4_ablation_prefill needs for `mode`: 0 for
 * MOE_W4_ABLATE_HOST_ROUTING, 3 * (E + 1) * I * H * 2 for
 * MOE_W4_ABLATE_SEPARATE_DEQUANT (0 also if the layer is invalid). */
size_t moe_w4_ablation_scratch_bytes(const moe_w4_layer* L, int mode);

/* moe_w4_forward_prefill with the variant `mode` (MOE_W4_ABLATE_*); same
 * arguments, layouts and ownership, plus `scratch`: device memory owned by the
 * caller, 16-byte aligned, at least moe_w4_ablation_scratch_bytes(L, mode)
 * bytes (unused, may be NULL, for MOE_W4_ABLATE_HOST_ROUTING).  Returns
 * MOE_W4_ERR_INVALID for an unknown mode or a missing scratch,
 * MOE_W4_ERR_ALIGN / MOE_W4_ERR_WORKSPACE for a misaligned or short scratch,
 * MOE_W4_ERR_DEVICE if a top-k index was out of range (host routing; nothing
 * written to `out`), the other codes as moe_w4_forward_prefill. */
int moe_w4_ablation_prefill(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out,
                            void* workspace, size_t ws_bytes, int mode, void* scratch, size_t scratch_bytes,
                            cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4_ABLATION_H */
