// Router of the prefill path: fp32 scores l[t,e] = sum_h x[t,h] W_r[h,e] (+bias)
// and, per token, the top-k experts with softmax weights over the selection
// plus the shared-expert gate sigmoid(x . g).
// ("Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three different workload shapes": score 256 experts per token, keep 8, one
// shared expert for every token.)
#include "common.cuh"
#include "internal.h"

namespace mw4 {

// ---------------------------------------------------------------------------
// scores: 64 tokens x 64 experts per CTA, 32-deep K slices, 4x4 per thread
// ---------------------------------------------------------------------------
constexpr int kRT = 64, kRE = 64, kRK = 32;

__global__ void __launch_bounds__(256) router_scores_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ Wr,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int T, int H, int E) {
    __shared__ float xs[kRK][kRT + 4];
    __shared__ __align__(16) float ws[kRK][kRE];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.y * kRT, e0 = blockIdx.x * kRE;
    const int ty = tid / 16, tx = tid % 16;
    float acc[4][4] = {};
    for (int h0 = 0; h0 < H; h0 += kRK) {
        {   // x tile: 64 tokens x 32 columns of bf16, one 16-byte load per thread
            const int t = tid / 4, c = (tid % 4) * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t0 + t < T) v = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * H + h0 + c);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xs[c + 2 * i][t] = __uint_as_float(u[i] << 16);
                xs[c + 2 * i + 1][t] = __uint_as_float(u[i] & 0xFFFF0000u);
            }
        }
        {   // W tile: 32 rows x 64 experts fp32
            const int r = tid / 8, c = (tid % 8) * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + c + i;
                ws[r][c + i] = (e < E) ? Wr[(size_t)(h0 + r) * E + e] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kRK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
            const float4 bv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
            b[0] = bv.x; b[1] = bv.y; b[2] = bv.z; b[3] = bv.w;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
        }
    }
}

// ---------------------------------------------------------------------------
// per-token selection: one warp per token
// ---------------------------------------------------------------------------
constexpr int kTopkWarps = 8;

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(const float* __restrict__ logits,
                                                               const uint16_t* __restrict__ x,
                                                               const float* __restrict__ g, int T, int H, int E,
                                                               int k, int32_t* __restrict__ idx,
                                                               float* __restrict__ w, float* __restrict__ gamma,
                                                               uint16_t* __restrict__ x16,
                                                               unsigned int* status) {
    extern __shared__ float sc_all[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    float* sc = sc_all + warp * E;
    for (int e = lane; e < E; e += 32) sc[e] = logits[(size_t)t * E + e];
    __syncwarp();
    select_topk_warp(sc, E, k, idx + (size_t)t * k, w + (size_t)t * k);
    float d = 0.f;
    for (int h = lane * 8; h < H; h += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)t * H + h);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t hv[4];
        bool fits = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = __uint_as_float(u[i] << 16), b = __uint_as_float(u[i] & 0xFFFF0000u);
            d = fmaf(a, g[h + 2 * i], d);
            d = fmaf(b, g[h + 2 * i + 1], d);
            fits = fits && fabsf(a) <= 65504.f && fabsf(b) <= 65504.f;
            hv[i] = h2_as_u32(__floats2half2_rn(a, b));
        }
        if (x16) {
            *reinterpret_cast<uint4*>(x16 + (size_t)t * H + h) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            if (!fits) raise_status(status, MOE_W4_STATUS_FP16_RANGE);
        }
    }
    d = warp_sum(d);
    if (lane == 0) gamma[t] = 1.0f / (1.0f + expf(-d));
}

cudaError_t launch_router_prefill(const moe_w4_layer& L, int T, const uint16_t* x, const RouteOut& o,
                                  cudaStream_t st) {
    dim3 grid((L.E + kRE - 1) / kRE, (T + kRT - 1) / kRT);
    router_scores_kernel<<<grid, 256, 0, st>>>(x, L.router_w, L.router_bias, o.logits, T, L.H, L.E);
    trace_mark(st, 1);
    const size_t sm = (size_t)kTopkWarps * L.E * sizeof(float);
    topk_kernel<<<(T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, sm, st>>>(
        o.logits, x, L.shared_gate, T, L.H, L.E, L.top_k, o.topk_idx, o.topk_w, o.gamma, o.x16, o.status);
    trace_mark(st, 2);
    return cudaGetLastError();
}

}  // namespace mw4
