// Measurement-only variant of the routing's grouping step: the expert
// histogram, the scan and the scatter computed on the host after the top-k
// indices are copied back, the way a CPU-synchronised routing step works.
// ("Optimizing on-device inference for Apple Silicon", section "Keep expert
// routing on the GPU": keeping the histogram, scan and scatter on the GPU
// avoids a round trip to the CPU between the router and the expert GEMMs.)
// The product path never calls this; moe_w4_ablation_prefill does, so that
// the cost of the round trip can be measured against the GPU-resident step.
// The records it writes are the ones the grouping kernels write: positions in
// token order within each expert, blocks of the tile's token rows, down units.
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace mw4 {

cudaError_t host_grouping(const moe_w4_layer& L, int T, const RouteOut& o, cudaStream_t st, bool* bad_index) {
    const int E = L.E, k = L.top_k, n = T * k;
    const TileCfg tc = tile_cfg(L, T);
    std::vector<int32_t> idx((size_t)n);
    cudaError_t e = cudaMemcpyAsync(idx.data(), o.topk_idx, (size_t)n * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    *bad_index = false;
    std::vector<int32_t> cnt((size_t)E, 0), off((size_t)E + 1, 0), perm((size_t)n), inv((size_t)n);
    for (int i = 0; i < n; ++i) {
        if (idx[i] < 0 || idx[i] >= E) { *bad_index = true; return cudaSuccess; }
        ++cnt[idx[i]];
    }
    for (int x = 0; x < E; ++x) off[x + 1] = off[x] + cnt[x];
    std::vector<int32_t> next(off.begin(), off.end() - 1);
    for (int i = 0; i < n; ++i) {   // i = t*k + j: token order within each expert
        const int p = next[idx[i]]++;
        perm[p] = i;
        inv[i] = p;
    }
    // blocks of bn rows per expert, then the shared group (every token, positions T*k ...)
    std::vector<int4> blk, uni;
    std::vector<int> first((size_t)E + 2, 0);
    for (int x = 0; x <= E; ++x) {
        first[x] = (int)blk.size();
        const int rows = x < E ? cnt[x] : T, p0 = x < E ? off[x] : n;
        for (int r0 = 0; r0 < rows; r0 += tc.bn) blk.push_back(make_int4(x, r0, std::min(tc.bn, rows - r0), p0 + r0));
    }
    first[E + 1] = (int)blk.size();
    for (int x = 0; x <= E; ++x) {
        const int b0 = first[x], nb = first[x + 1] - b0;
        for (int j = 0; j * tc.du < nb; ++j) uni.push_back(make_int4(b0 + j * tc.du, std::min(tc.du, nb - j * tc.du), x, 0));
    }
    const int32_t nt[2] = {(int32_t)blk.size() * (L.I / kBM), (int32_t)uni.size() * (L.H / kBM)};
    e = cudaMemcpyAsync(o.counts, cnt.data(), (size_t)E * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o.offsets, off.data(), ((size_t)E + 1) * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o.perm, perm.data(), (size_t)n * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o.inv, inv.data(), (size_t)n * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o.blkinfo, blk.data(), blk.size() * sizeof(int4), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o.unitinfo, uni.data(), uni.size() * sizeof(int4), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o.ntiles, nt, sizeof(nt), cudaMemcpyHostToDevice, st);
    // the host vectors must outlive the copies
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

}  // namespace mw4

namespace mw4 {

// ---------------------------------------------------------------------------
// Separate dequantisation pass: the layer's weights rebuilt in fp16 in memory,
// for the grouped GEMMs to read back.  ("Optimizing on-device inference for
// Apple Silicon", section "Dequantise weights during matrix multiplication":
// expanding the 4-bit weights to a 16-bit array that the matmul then reads is
// what the fused dequantisation replaces.)  Each weight is the value the fused
// dequantisers put in tensor memory (same fp16 roundings), at the same K
// position (chunk order), so the variant's output equals the product's.
// ---------------------------------------------------------------------------
template <int BITS, bool E4M3>
__global__ void __launch_bounds__(256) f16_weights_kernel(const uint32_t* __restrict__ codes,
                                                          const uint16_t* __restrict__ sc,
                                                          const uint16_t* __restrict__ bi, size_t rows, int cols,
                                                          uint16_t* __restrict__ out, unsigned int* status) {
    constexpr int kPerWord = 32 / BITS;   // columns per code word
    const int wpr = cols / kPerWord, G = cols / kGroup;
    const size_t n = rows * (size_t)wpr;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / wpr;
        const int col0 = (int)(i % wpr) * kPerWord, g = col0 / kGroup;
        const float sf = bf16_bits_to_float(sc[r * G + g]), bf = bf16_bits_to_float(bi[r * G + g]);
        constexpr float kQmax = BITS == 4 ? 15.f : (E4M3 ? 448.f : 255.f);
        if (!(fmaf(fabsf(sf), kQmax, fabsf(bf)) <= 65504.f)) raise_status(status, MOE_W4_STATUS_FP16_RANGE);
        const __half s_h = __float2half_rn(sf), s_h16 = __float2half_rn(sf * 0.0625f), b_h = __float2half_rn(bf);
        const __half2 s2 = __halves2half2(s_h, s_h), s2_16 = __halves2half2(s_h16, s_h16), b2 = __halves2half2(b_h, b_h);
        const uint32_t w = codes[i];
        uint16_t* dst = out + r * cols + col0;
        if (BITS == 4) {
            uint32_t o[4];
            dequant8_f16(w, s2, s2_16, b2, o);
            *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            uint32_t o[2];
            if (E4M3)
                dequant_e4m3x4_f16(w, s2, b2, o);
            else
                dequant4x8_f16(w, s2, b2, o);
            *reinterpret_cast<uint2*>(dst) = make_uint2(o[0], o[1]);
        }
    }
}

size_t f16_weights_bytes(const moe_w4_layer& L) {
    return 3 * ((size_t)L.E + 1) * (size_t)L.I * (size_t)L.H * 2;
}

cudaError_t launch_f16_weights(const moe_w4_layer& L, uint16_t* w16, const uint16_t* w16_ptrs[6], unsigned int* status,
                               cudaStream_t st) {
    const size_t E = L.E, H = L.H, I = L.I;
    const moe_w4_mat* ms[6] = {&L.gate, &L.up, &L.down, &L.sh_gate, &L.sh_up, &L.sh_down};
    const size_t rows[6] = {E * I, E * I, E * H, I, I, H};
    const int cols[6] = {(int)H, (int)H, (int)I, (int)H, (int)H, (int)I};
    const int bits = code_bits_of(L);
    const bool e4m3 = codes_e4m3(L);
    uint16_t* o = w16;
    for (int m = 0; m < 6; ++m) {
        w16_ptrs[m] = o;
        const size_t words = rows[m] * (size_t)cols[m] * bits / 32;
        const unsigned grid = (unsigned)std::min<size_t>((words + 255) / 256, 152 * 8);
        if (bits == 4)
            f16_weights_kernel<4, false><<<grid, 256, 0, st>>>(ms[m]->codes, ms[m]->scales, ms[m]->biases, rows[m],
                                                               cols[m], o, status);
        else if (e4m3)
            f16_weights_kernel<8, true><<<grid, 256, 0, st>>>(ms[m]->codes, ms[m]->scales, ms[m]->biases, rows[m],
                                                              cols[m], o, status);
        else
            f16_weights_kernel<8, false><<<grid, 256, 0, st>>>(ms[m]->codes, ms[m]->scales, ms[m]->biases, rows[m],
                                                               cols[m], o, status);
        o += rows[m] * (size_t)cols[m];
    }
    return cudaGetLastError();
}

}  // namespace mw4
