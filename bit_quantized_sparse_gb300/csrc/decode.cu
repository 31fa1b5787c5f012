// Decode path (1 <= T <= 16 tokens): every weight is read once per token-expert
// pair, so the path is bound by HBM reads of the packed codes.
// ("Optimizing on-device inference for Apple Silicon", sections "Optimise the
// single-row weight path" -- row-parallel GEMV, groups of threads cooperating
// on outputs while reading different parts of the weight matrix -- and "Reduce
// intermediate state and traffic" -- gate and up projections fused with the
// gated activation; output projection fused with the routing scores and the
// shared expert's result.)
//
// The allocation-free entry point runs these when the fused batch-1 kernel
// does not cover the layer (or its cooperative launch is refused).  Three
// kernels on one stream, no host round trip:
//   1. decode_router_kernel  partial scores over 256-row slices of W_r; the
//      last CTA to finish (atomic ticket, no spinning) reduces them in a fixed
//      order, selects the top-k, the softmax weights and the shared gate.
//   2. decode_gateup_kernel  one warp per (token, expert, 2 rows): gate and up
//      rows dequantised in registers, SwiGLU, h in fp32.
//   3. decode_down_kernel    one warp per (token, 8 output rows): the down rows
//      of all k+1 experts, weighted and summed in-register, bf16 out.
#include "common.cuh"
#include "internal.h"

namespace mw4 {

__global__ void __launch_bounds__(256) decode_router_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ Wr,
                                                            const float* __restrict__ bias,
                                                            const float* __restrict__ g, int T, int H, int E,
                                                            int k, DecodeWs d) {
    __shared__ float red[8][kDecodeMaxT][32];
    __shared__ int is_last;
    extern __shared__ float sc_all[];   // [8][E] in the last CTA
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int e = blockIdx.x * 32 + lane;
    const int h0 = blockIdx.y * kRouterRowsPerCta;
    float acc[kDecodeMaxT];
#pragma unroll
    for (int t = 0; t < kDecodeMaxT; ++t) acc[t] = 0.f;
    for (int r = warp; r < kRouterRowsPerCta && h0 + r < H; r += 8) {
        const int h = h0 + r;
        const float wv = (e < E) ? __ldg(Wr + (size_t)h * E + e) : 0.f;
#pragma unroll
        for (int t = 0; t < kDecodeMaxT; ++t)
            if (t < T) acc[t] = fmaf(bf16_bits_to_float(x[(size_t)t * H + h]), wv, acc[t]);
    }
#pragma unroll
    for (int t = 0; t < kDecodeMaxT; ++t) red[warp][t][lane] = acc[t];
    __syncthreads();
    for (int i = tid; i < T * 32; i += blockDim.x) {
        const int t = i / 32, l = i % 32, ee = blockIdx.x * 32 + l;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w][t][l];
        if (ee < E) d.part[((size_t)blockIdx.y * T + t) * E + ee] = s;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned int nblk = gridDim.x * gridDim.y;
        is_last = (atomicAdd(d.counter, 1u) == nblk - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // last CTA: fixed-order reduction over the row slices, then selection
    const int nslice = gridDim.y;
    for (int t = warp; t < T; t += 8) {
        float* sc = sc_all + warp * E;
        for (int ee = lane; ee < E; ee += 32) {
            float s = 0.f;
            for (int sl = 0; sl < nslice; ++sl) s += __ldcg(d.part + ((size_t)sl * T + t) * E + ee);
            sc[ee] = s + (bias ? bias[ee] : 0.f);
        }
        __syncwarp();
        select_topk_warp(sc, E, k, d.idx + (size_t)t * k, d.w + (size_t)t * k);
        float dd = 0.f;
        for (int h = lane; h < H; h += 32) dd = fmaf(bf16_bits_to_float(x[(size_t)t * H + h]), g[h], dd);
        dd = warp_sum(dd);
        if (lane == 0) d.gamma[t] = 1.0f / (1.0f + expf(-dd));
        __syncwarp();
    }
    if (tid == 0) *d.counter = 0u;   // ready for the next call
}

// Dot product of 32 input columns (4 code words) with x: s * sum(q x) + b * sum(x).
MW4_DEV float w4_dot32(const uint4 cw, float s, float b, const float* xs) {
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
    float sqx = 0.f, sx = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const float xv = xs[i * 8 + n];
            sqx = fmaf((float)((w[i] >> (4 * n)) & 15u), xv, sqx);
            sx += xv;
        }
    }
    return fmaf(s, sqx, b * sx);
}

struct MatPtrs { const uint32_t* codes; const uint16_t* s; const uint16_t* b; };

MW4_DEV MatPtrs expert_mat(const moe_w4_mat& routed, const moe_w4_mat& shared, int e, int E, size_t rows,
                           size_t cols) {
    if (e >= E) return {shared.codes, shared.scales, shared.biases};
    return {routed.codes + (size_t)e * rows * (cols / 8), routed.scales + (size_t)e * rows * (cols / kGroup),
            routed.biases + (size_t)e * rows * (cols / kGroup)};
}

constexpr int kGU_Warps = 16, kGU_RowsPerWarp = 2, kGU_Rows = kGU_Warps * kGU_RowsPerWarp;

__global__ void __launch_bounds__(kGU_Warps * 32) decode_gateup_kernel(moe_w4_layer L, const uint16_t* __restrict__ x,
                                                                      DecodeWs d) {
    extern __shared__ float xf[];   // [H]
    const int H = L.H, I = L.I, E = L.E, k = L.top_k;
    const int slot = blockIdx.y, t = blockIdx.z;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int h = tid; h < H; h += blockDim.x) xf[h] = bf16_bits_to_float(x[(size_t)t * H + h]);
    const int e = (slot < k) ? d.idx[t * k + slot] : E;
    __syncthreads();
    if (e < 0 || e > E) { if (tid == 0) raise_status(d.status, MOE_W4_STATUS_BAD_INDEX); return; }
    const MatPtrs G = expert_mat(L.gate, L.sh_gate, e, E, I, H);
    const MatPtrs U = expert_mat(L.up, L.sh_up, e, E, I, H);
    const int W = H / 8, NG = H / kGroup;
    float ag[kGU_RowsPerWarp] = {}, au[kGU_RowsPerWarp] = {};
    const int i0 = blockIdx.x * kGU_Rows + warp * kGU_RowsPerWarp;
    for (int w0 = lane * 4; w0 < W; w0 += 128) {
        const int grp = w0 / 8;
        uint4 cg[kGU_RowsPerWarp], cu[kGU_RowsPerWarp];
#pragma unroll
        for (int r = 0; r < kGU_RowsPerWarp; ++r) {
            cg[r] = __ldg(reinterpret_cast<const uint4*>(G.codes + (size_t)(i0 + r) * W + w0));
            cu[r] = __ldg(reinterpret_cast<const uint4*>(U.codes + (size_t)(i0 + r) * W + w0));
        }
#pragma unroll
        for (int r = 0; r < kGU_RowsPerWarp; ++r) {
            const size_t gi = (size_t)(i0 + r) * NG + grp;
            ag[r] += w4_dot32(cg[r], bf16_bits_to_float(G.s[gi]), bf16_bits_to_float(G.b[gi]), xf + w0 * 8);
            au[r] += w4_dot32(cu[r], bf16_bits_to_float(U.s[gi]), bf16_bits_to_float(U.b[gi]), xf + w0 * 8);
        }
    }
#pragma unroll
    for (int r = 0; r < kGU_RowsPerWarp; ++r) {
        const float gs = warp_sum(ag[r]), us = warp_sum(au[r]);
        if (lane == 0) d.hh[((size_t)t * (k + 1) + slot) * I + i0 + r] = silu_f(gs) * us;
    }
}

constexpr int kDN_Warps = 8, kDN_RowsPerWarp = 8, kDN_Rows = kDN_Warps * kDN_RowsPerWarp;

__global__ void __launch_bounds__(kDN_Warps * 32) decode_down_kernel(moe_w4_layer L, uint16_t* __restrict__ out,
                                                                    DecodeWs d) {
    extern __shared__ float hs[];   // [(k+1)][I]
    __shared__ int es[9];
    __shared__ float wts[9];
    const int H = L.H, I = L.I, E = L.E, k = L.top_k;
    const int t = blockIdx.y;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < (k + 1) * I; i += blockDim.x) hs[i] = d.hh[(size_t)t * (k + 1) * I + i];
    if (tid <= k) {
        es[tid] = (tid < k) ? d.idx[t * k + tid] : E;
        wts[tid] = (tid < k) ? d.w[t * k + tid] : d.gamma[t];
    }
    __syncthreads();
    const int W = I / 8, NG = I / kGroup;
    for (int r = 0; r < kDN_RowsPerWarp; ++r) {
        const int o = blockIdx.x * kDN_Rows + warp * kDN_RowsPerWarp + r;
        float acc = 0.f;
        for (int slot = 0; slot <= k; ++slot) {
            const int e = es[slot];
            if (e < 0 || e > E) continue;
            const MatPtrs D = expert_mat(L.down, L.sh_down, e, E, H, I);
            const float* hv = hs + slot * I;
            float part = 0.f;
            for (int w0 = lane * 2; w0 < W; w0 += 64) {
                const uint2 cw = __ldg(reinterpret_cast<const uint2*>(D.codes + (size_t)o * W + w0));
                const size_t gi = (size_t)o * NG + w0 / 8;
                const float s = bf16_bits_to_float(D.s[gi]), b = bf16_bits_to_float(D.b[gi]);
                const uint32_t cws[2] = {cw.x, cw.y};
                float sqh = 0.f, sh = 0.f;
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int n = 0; n < 8; ++n) {
                        const float h = hv[(w0 + i) * 8 + n];
                        sqh = fmaf((float)((cws[i] >> (4 * n)) & 15u), h, sqh);
                        sh += h;
                    }
                part += fmaf(s, sqh, b * sh);
            }
            acc = fmaf(wts[slot], part, acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) out[(size_t)t * H + o] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
}

// The rows of a T-row call that may go through the one-kernel path (T unless
// the moe_w4_test_refuse_fused_after hook is on; defined with it in api.cu); the
// rest take the fallback of a refused cooperative launch.
int test_fused_rows_allowed(int T);

cudaError_t launch_decode(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out, const DecodeWs& d_in,
                          cudaStream_t st) {
    const int k = L.top_k;
    DecodeWs d = d_in;
    if (decode_fused_supported(L)) {   // one launch per row for the whole layer
        const int done = launch_decode_fused_rows(L, test_fused_rows_allowed(T), x, out, d, st);
        if (done == T) return cudaGetLastError();
        // a launch was refused (the grid cannot be resident at once): the rows not
        // yet enqueued take the three kernels below, which read 4-bit codes only
        if (code_bits_of(L) != 4) return cudaErrorNotSupported;
        x += (size_t)done * L.H;
        out += (size_t)done * L.H;
        d.idx += (size_t)done * k;
        d.w += (size_t)done * k;
        d.gamma += done;
        T -= done;
    }
    static bool attrs_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attrs_set[dev]) {   // the largest sizes any supported shape needs
        cudaFuncSetAttribute(decode_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 * 1024 * 4);
        cudaFuncSetAttribute(decode_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 4096 * 4);
        cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 9 * 4096 * 4);
        attrs_set[dev] = true;
    }
    trace_kernels(3);
    dim3 g1((L.E + 31) / 32, (L.H + kRouterRowsPerCta - 1) / kRouterRowsPerCta);
    decode_router_kernel<<<g1, 256, 8 * L.E * sizeof(float), st>>>(x, L.router_w, L.router_bias, L.shared_gate, T,
                                                                   L.H, L.E, k, d);
    trace_mark(st, 1);
    dim3 g2(L.I / kGU_Rows, k + 1, T);
    decode_gateup_kernel<<<g2, kGU_Warps * 32, L.H * sizeof(float), st>>>(L, x, d);
    trace_mark(st, 2);
    dim3 g3(L.H / kDN_Rows, T);
    decode_down_kernel<<<g3, kDN_Warps * 32, (k + 1) * L.I * sizeof(float), st>>>(L, out, d);
    trace_mark(st, 3);
    return cudaGetLastError();
}

}  // namespace mw4
