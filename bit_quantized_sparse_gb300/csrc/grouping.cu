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

// chunk_base[c][e] <- number of assignments to e in tokens [c*kChunk, (c+1)*kChunk)
__global__ void __launch_bounds__(kChunk) chunk_count_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                             int32_t* __restrict__ chunk_base,
                                                             unsigned int* status) {
    extern __shared__ int hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * kChunk + threadIdx.x;
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = idx[(size_t)t * k + j];
            if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
            else raise_status(status, MOE_W4_STATUS_BAD_INDEX);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_base[(size_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan of n <= 2*blockDim values in shared memory `a` (in place);
// returns the total.  blockDim is a multiple of 32.
__device__ int block_exclusive_scan(int* a, int n, int* warp_tot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int i0 = 2 * tid;
    const int v0 = (i0 < n) ? a[i0] : 0, v1 = (i0 + 1 < n) ? a[i0 + 1] : 0;
    int s = v0 + v1, incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = (lane < nw) ? warp_tot[lane] : 0, wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < nw) warp_tot[lane] = wi - wv;   // exclusive warp prefix
        if (lane == 31) warp_tot[32] = wi;          // total
    }
    __syncthreads();
    const int excl = warp_tot[warp] + incl - s;
    if (i0 < n) a[i0] = excl;
    if (i0 + 1 < n) a[i0 + 1] = excl + v0;
    const int total = warp_tot[32];
    __syncthreads();
    return total;
}

// One CTA: per-expert totals over chunks (chunk_base becomes the absolute
// start of each chunk inside its expert group), expert offsets, and the tile
// lists of the grouped GEMMs (expert-major, then row block, then weight block).
constexpr int kScanRegChunks = 32;   // chunk counts held in registers (T <= 32 * kChunk)

__global__ void __launch_bounds__(1024) scan_kernel(int T, int E, int k, int nchunk, int32_t* __restrict__ chunk_base,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int4* __restrict__ blkinfo, int4* __restrict__ unitinfo,
                                                    int32_t* __restrict__ ntiles, int MI, int MH, int R, int BN) {
    extern __shared__ int sm[];
    int* cnt = sm;               // [E+1]
    int* off = sm + (E + 1);     // [E+1]
    int* blk = off + (E + 1);    // [E+1]
    int* uni = blk + (E + 1);    // [E+1]
    int* wt = uni + (E + 1);     // [33]
    // up to kScanRegChunks chunks: the counts of one expert stay in registers as
    // exclusive prefixes and are written once, offset added, after the scan
    const bool in_regs = nchunk <= kScanRegChunks;
    int pre[kScanRegChunks];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        if (in_regs) {
#pragma unroll
            for (int j = 0; j < kScanRegChunks; ++j) pre[j] = (j < nchunk) ? chunk_base[(size_t)j * E + e] : 0;
#pragma unroll
            for (int j = 0; j < kScanRegChunks; ++j) {
                const int c = pre[j];
                pre[j] = run;
                run += c;
            }
        } else {
            for (int c0 = 0; c0 < nchunk; c0 += 8) {   // eight independent loads in flight
                int v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = (c0 + j < nchunk) ? chunk_base[(size_t)(c0 + j) * E + e] : 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (c0 + j < nchunk) chunk_base[(size_t)(c0 + j) * E + e] = run;
                    run += v[j];
                }
            }
        }
        cnt[e] = run;
        off[e] = run;
        blk[e] = (run + BN - 1) / BN;
    }
    if (threadIdx.x == 0) {
        cnt[E] = T;                        // shared expert: every token, in order
        off[E] = T;
        blk[E] = (T + BN - 1) / BN;
    }
    __syncthreads();
    block_exclusive_scan(off, E + 1, wt);      // off[e] = start of group e; off[E] = T*k
    const int nblk = block_exclusive_scan(blk, E + 1, wt);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        counts[e] = cnt[e];
        offsets[e] = off[e];
        if (in_regs) {
            // E <= 1024 = blockDim.x: each thread owns at most one expert, whose prefixes pre[] holds
#pragma unroll
            for (int j = 0; j < kScanRegChunks; ++j)
                if (j < nchunk) chunk_base[(size_t)j * E + e] = pre[j] + off[e];
        } else {
            for (int c = 0; c < nchunk; ++c) chunk_base[(size_t)c * E + e] += off[e];
        }
    }
    if (threadIdx.x == 0) offsets[E] = off[E];
    if (blkinfo == nullptr) return;
    // one record per block of BN rows (128 unless a tile override is set): the GEMMs read their tile's block in one load
    // (tile = block * M + weight-row block); the shared group (e = E) comes last
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        const int b0 = blk[e], b1 = (e < E) ? blk[e + 1] : nblk;
        const int rows = (e < E) ? cnt[e] : T, p_first = (e < E) ? off[e] : T * k;
        for (int b = b0; b < b1; ++b) {
            const int r0 = (b - b0) * BN;
            blkinfo[b] = make_int4(e, r0, min(BN, rows - r0), p_first + r0);
        }
    }
    // down units: runs of at most R consecutive row blocks of one group
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        const int nb = ((e < E) ? blk[e + 1] : nblk) - blk[e];
        uni[e] = (nb + R - 1) / R;
    }
    __syncthreads();
    const int nuni = block_exclusive_scan(uni, E + 1, wt);
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        const int b0 = blk[e], nb = ((e < E) ? blk[e + 1] : nblk) - b0;
        for (int j = 0; j * R < nb; ++j) unitinfo[uni[e] + j] = make_int4(b0 + j * R, min(R, nb - j * R), e, 0);
    }
    if (threadIdx.x == 0) {
        ntiles[0] = nblk * MI;
        ntiles[1] = nuni * MH;
    }
}

// One warp per chunk walks its tokens in order and gives every assignment its
// grouped position; lanes holding the same expert in one step are ranked by
// lane order, which is token order.
// Four warps per chunk of kChunk tokens, warp w taking tokens [32w, 32w+32):
// each warp first counts its tokens' selections per expert, the counts are
// turned into per-warp starting positions (chunk base + earlier warps'
// counts), then every warp places its own tokens in order.  Positions are
// therefore the same as one warp walking the whole chunk in token order.
constexpr int kAssignWarps = kChunk / 32;
__global__ void __launch_bounds__(kChunk) assign_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                                        const int32_t* __restrict__ chunk_base,
                                                        int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                                        unsigned int* status) {
    extern __shared__ int sm_assign[];
    int* running = sm_assign;                       // [kAssignWarps][E]
    int* sel = sm_assign + kAssignWarps * E;        // [kChunk * k] the chunk's selections
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x;
    const int t_begin = c * kChunk, t_end = min(T, t_begin + kChunk);
    for (int i = threadIdx.x; i < kAssignWarps * E; i += blockDim.x) running[i] = 0;
    for (int i = threadIdx.x; i < (t_end - t_begin) * k; i += blockDim.x) sel[i] = idx[(size_t)t_begin * k + i];
    __syncthreads();
    const int w_begin = min(t_end, t_begin + 32 * warp), w_end = min(t_end, w_begin + 32);
    int* run_w = running + warp * E;
    for (int i = lane; i < (w_end - w_begin) * k; i += 32) {   // this warp's counts
        const int e = sel[(w_begin - t_begin) * k + i];
        if (e >= 0 && e < E) atomicAdd(&run_w[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {    // counts -> starting positions
        int base = chunk_base[(size_t)c * E + e];
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
        if (e < 0 || e >= E) e = -1;        // bad indices were reported by the count kernel
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

cudaError_t launch_grouping(const moe_w4_layer& L, int T, const RouteOut& o, cudaStream_t st, const TileCfg* force) {
    const int E = L.E, k = L.top_k;
    const int nchunk = (T + kChunk - 1) / kChunk;
    chunk_count_kernel<<<nchunk, kChunk, E * sizeof(int), st>>>(o.topk_idx, T, E, k, o.chunk_base, o.status);
    trace_mark(st, 3);
    const size_t scan_sm = (4 * (E + 1) + 33) * sizeof(int);
    const TileCfg tc = force ? *force : tile_cfg(L, T);
    scan_kernel<<<1, 1024, scan_sm, st>>>(T, E, k, nchunk, o.chunk_base, o.counts, o.offsets, o.blkinfo, o.unitinfo,
                                          o.ntiles, L.I / kBM, L.H / kBM, tc.du, tc.bn);
    trace_mark(st, 4);
    assign_kernel<<<nchunk, kChunk, (kAssignWarps * E + kChunk * k) * sizeof(int), st>>>(o.topk_idx, T, E, k, o.chunk_base, o.perm,
                                                                     o.inv, o.status);
    trace_mark(st, 5);
    return cudaGetLastError();
}

}  // namespace mw4
