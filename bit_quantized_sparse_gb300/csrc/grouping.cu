// Expert grouping on the GPU: per-chunk histograms of the assignments, one
// prefix scan to expert offsets (plus the block lists the grouped GEMMs walk),
// and a stable scatter giving each assignment its grouped position.
// ("Optimizing on-device inference for Apple Silicon", section "Keep expert
// routing on the GPU": histogram -> prefix scan -> scatter -> block map, all
// enqueued without a CPU round trip.)
//
// Determinism: the position of assignment (t, j) of expert e is
// offsets[e] + #{t' < t : t' selected e}; chunks are scanned in token order
// and, inside a chunk, one warp walks the tokens in order, so no result
// depends on atomic ordering.
#include "common.cuh"
#include "internal.h"

namespace mw4 {

// Exclusive scan of a[0..n) in shared memory (in place) by the whole block, any
// n: each thread scans a contiguous segment, the segment totals are scanned by
// warp shuffles through `wt` (at least 33 ints); returns the total.
__device__ int block_scan_excl(int* a, int n, int* wt) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x, i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int s = 0;
    for (int i = i0; i < i1; ++i) s += a[i];
    int incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) wt[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int wv = lane < nw ? wt[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < nw) wt[lane] = wi - wv;   // exclusive warp prefix
        if (lane == 31) wt[32] = wi;         // total
    }
    __syncthreads();
    int run = wt[warp] + incl - s;
    for (int i = i0; i < i1; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    const int total = wt[32];
    __syncthreads();
    return total;
}

// The whole grouping in one launch, one CTA per chunk of kChunk tokens
// (kChunk threads).  The top-k kernel has counted each chunk's assignments
// per expert (hist[c][e]).  Every CTA forms the expert totals, their
// exclusive scan (the expert offsets), the block and unit counts per group and
// their scans, and the start of its own chunk inside each expert group
// (offset + the earlier chunks' counts).  It writes the grouped GEMMs' records
// for its share of the groups: blocks of BN rows per expert group (the shared
// expert's group, every token, last) and down units of at most R blocks; CTA 0
// writes counts, offsets and the tile counts.  Its four warps then give the
// chunk's assignments their grouped positions in token order: warp w takes
// tokens [32w, 32w+32), counts its selections per expert, the counts become
// per-warp starting positions (chunk start + earlier warps' counts), and each
// warp places its own tokens, lanes holding the same expert ranked by lane
// order (token order).  Positions are therefore offsets[e] + the number of
// earlier tokens that chose e.
constexpr int kAssignWarps = kChunk / 32;
constexpr int kHistSplit = 2;     // chunk halves summed by separate threads (loads in flight)
constexpr int kHistLoads = 16;    // 16-byte histogram loads in flight per thread
__global__ void __launch_bounds__(kChunk) group_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                       int nchunk, const int32_t* __restrict__ hist,
                                                       int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                       int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                                       int4* __restrict__ blkinfo, int4* __restrict__ unitinfo,
                                                       int32_t* __restrict__ ntiles, int MI, int MH, int R, int BN,
                                                       unsigned int* status) {
    griddep_wait();               // programmatic dependent launch: nothing is touched before the
    griddep_launch_dependents();  // previous kernel has completed; the next one may be scheduled
    extern __shared__ int sm_group[];
    int* off = sm_group;                     // [E+1] totals, then their exclusive scan
    int* start = off + (E + 1);              // [E] this chunk's start inside each group
    int* running = start + E;                // [kAssignWarps][E]; first the chunk-half sums [2][2][E]
    int* sel = running + kAssignWarps * E;   // [kChunk * k] the chunk's selections
    int* wt = sel + kChunk * k;              // [64] scan scratch
    int* blk = wt + 64;                      // [E+1] blocks per group, then the first block of each
    int* uni = blk + (E + 1);                // [E+1] units per group, then the first unit of each
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, c = blockIdx.x;
    const int t_begin = c * kChunk, t_end = min(T, t_begin + kChunk);
    for (int i = threadIdx.x; i < (t_end - t_begin) * k; i += blockDim.x) sel[i] = idx[(size_t)t_begin * k + i];
    // totals and this chunk's prefix: thread (h, q) sums experts [4q, 4q+4) (one
    // expert q if E is not a multiple of 4) over the chunks of half h, kHistLoads
    // loads in flight
    {
        int* part = running;   // [kHistSplit][2][E]: totals and prefixes of each half
        const bool vec = (E % 4) == 0;
        const int nq = vec ? E / 4 : E, nchalf = (nchunk + kHistSplit - 1) / kHistSplit;
        for (int w = threadIdx.x; w < kHistSplit * nq; w += blockDim.x) {
            const int h = w / nq, q = w % nq, c0 = h * nchalf, c1 = min(nchunk, c0 + nchalf);
            int4 tot = make_int4(0, 0, 0, 0), pre = tot;
            for (int cb = c0; cb < c1; cb += kHistLoads) {
                int4 v[kHistLoads];
#pragma unroll
                for (int j = 0; j < kHistLoads; ++j) {
                    const int32_t* row = hist + (size_t)(cb + j) * E;
                    v[j] = cb + j >= c1 ? make_int4(0, 0, 0, 0)
                         : vec          ? reinterpret_cast<const int4*>(row)[q]
                                        : make_int4(row[q], 0, 0, 0);
                }
#pragma unroll
                for (int j = 0; j < kHistLoads; ++j) {
                    if (cb + j == c) pre = tot;
                    tot.x += v[j].x; tot.y += v[j].y; tot.z += v[j].z; tot.w += v[j].w;
                }
            }
            if (c >= c1) pre = tot;           // every chunk of this half precedes c
            int* pt = part + h * 2 * E;
            int* pp = pt + E;
            if (vec) {
                pt[4 * q] = tot.x; pt[4 * q + 1] = tot.y; pt[4 * q + 2] = tot.z; pt[4 * q + 3] = tot.w;
                pp[4 * q] = pre.x; pp[4 * q + 1] = pre.y; pp[4 * q + 2] = pre.z; pp[4 * q + 3] = pre.w;
            } else {
                pt[q] = tot.x;
                pp[q] = pre.x;
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int tot = 0, pre = 0;
#pragma unroll
            for (int h = 0; h < kHistSplit; ++h) {   // halves in chunk order
                const int* pt = part + h * 2 * E;
                pre += (h * nchalf <= c) ? pt[E + e] : 0;
                tot += pt[e];
            }
            off[e] = tot;
            start[e] = pre;
        }
    }
    if (threadIdx.x == 0) off[E] = 0;
    __syncthreads();
    if (c == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = off[e];
    block_scan_excl(off, E + 1, wt);   // off[e] = start of group e; off[E] = T*k
    for (int e = threadIdx.x; e < E; e += blockDim.x) start[e] += off[e];
    if (c == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off[e];
    if (blkinfo != nullptr) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) blk[e] = ((e < E ? off[e + 1] - off[e] : T) + BN - 1) / BN;
        __syncthreads();
        const int nblk = block_scan_excl(blk, E + 1, wt);
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            const int nb = (e < E ? blk[e + 1] : nblk) - blk[e];
            uni[e] = (nb + R - 1) / R;
        }
        __syncthreads();
        const int nuni = block_scan_excl(uni, E + 1, wt);
        // this CTA's share of the groups: e = c, c + nchunk, ...
        for (int e = c + (int)threadIdx.x * nchunk; e <= E; e += (int)blockDim.x * nchunk) {
            const int b0 = blk[e], nb = (e < E ? blk[e + 1] : nblk) - b0;
            const int rows = e < E ? off[e + 1] - off[e] : T, p_first = e < E ? off[e] : T * k;
            for (int b = 0; b < nb; ++b) {
                const int r0 = b * BN;
                blkinfo[b0 + b] = make_int4(e, r0, min(BN, rows - r0), p_first + r0);
            }
            for (int j = 0; j * R < nb; ++j) unitinfo[uni[e] + j] = make_int4(b0 + j * R, min(R, nb - j * R), e, 0);
        }
        if (c == 0 && threadIdx.x == 0) {
            ntiles[0] = nblk * MI;
            ntiles[1] = nuni * MH;
        }
    }
    for (int i = threadIdx.x; i < kAssignWarps * E; i += blockDim.x) running[i] = 0;
    __syncthreads();
    // the assignments of this chunk, in token order
    const int w_begin = min(t_end, t_begin + 32 * warp), w_end = min(t_end, w_begin + 32);
    int* run_w = running + warp * E;
    for (int i = lane; i < (w_end - w_begin) * k; i += 32) {   // this warp's counts
        const int e = sel[(w_begin - t_begin) * k + i];
        if (e >= 0 && e < E) atomicAdd(&run_w[e], 1);
        else raise_status(status, MOE_W4_STATUS_BAD_INDEX);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {    // counts -> starting positions
        int base = start[e];
#pragma unroll
        for (int w = 0; w < kAssignWarps; ++w) {
            const int n = running[w * E + e];
            running[w * E + e] = base;
            base += n;
        }
    }
    __syncthreads();
    const int per = 32 / k;                 // tokens per step
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int t0 = w_begin; t0 < w_end; t0 += per) {
        const int t = t0 + lane / k, j = lane % k;
        const bool valid = (lane < per * k) && (t < w_end);
        int e = valid ? sel[(t - t_begin) * k + j] : -1;
        if (e < 0 || e >= E) e = -1;        // reported above
        const unsigned same = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = run_w[e] + __popc(same & lt_mask);
        __syncwarp();
        if (e >= 0 && (same & lt_mask) == 0) run_w[e] += __popc(same);   // group leader
        __syncwarp();
        if (e >= 0) {
            pos = checked_index(pos, 0, T * k, status);
            perm[pos] = t * k + j;
            inv[(size_t)t * k + j] = pos;
        }
    }
}

// Shared memory of group_kernel.
static size_t group_smem(int E, int k) {
    return ((size_t)(E + 1) + E + (size_t)kAssignWarps * E + (size_t)kChunk * k + 64 + 2 * (E + 1)) * sizeof(int);
}

cudaError_t launch_grouping(const moe_w4_layer& L, int T, const RouteOut& o, cudaStream_t st, const TileCfg* force) {
    const int E = L.E, k = L.top_k;
    const int nchunk = (T + kChunk - 1) / kChunk;
    const TileCfg tc = force ? *force : tile_cfg(L, T);
    const size_t sm = group_smem(E, k);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {   // the largest: E = 1024, k = 8
        const cudaError_t e = cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)group_smem(1024, 8));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const cudaError_t e = launch_pdl(pdl_for(T), group_kernel, dim3(nchunk), dim3(kChunk), sm, st, o.topk_idx, T, E, k, nchunk,
                                     o.chunk_base, o.counts, o.offsets, o.perm, o.inv, o.blkinfo, o.unitinfo, o.ntiles,
                                     L.I / kBM, L.H / kBM, tc.du, tc.bn, o.status);
    if (e != cudaSuccess) return e;
    trace_mark(st, 3);
    return cudaGetLastError();
}

}  // namespace mw4
