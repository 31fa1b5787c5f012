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
