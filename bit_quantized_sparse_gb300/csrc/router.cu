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
// scores on the tensor cores with fp32 accuracy
// ---------------------------------------------------------------------------
// W_r (fp32) is split exactly into three bf16 terms, w = hi + mid + lo (8 + 8 +
// 8 significant bits), stored transposed as A[e][k] for k in [0, 3H): hi, then
// mid, then lo.  x is exact in bf16, every bf16 x bf16 product is exact in
// fp32, and the tensor core accumulates in fp32, so A . [x, x, x] reproduces
// the fp32 score x . W_r.  Rows e >= E are zero.
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ Wr, int H, int E, int Epad,
                                                           uint16_t* __restrict__ A) {
    __shared__ float tile[32][33];
    const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;   // 32 x 8
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + tx;
        tile[r][tx] = (e < E) ? Wr[(size_t)(h0 + r) * E + e] : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {   // r: expert within the tile, tx: row h within the tile
        const int e = e0 + r;
        if (e >= Epad) continue;
        const float w = tile[tx][r];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        uint16_t* row = A + (size_t)e * 3 * H + h0 + tx;
        row[0] = __bfloat16_as_ushort(hi);
        row[H] = __bfloat16_as_ushort(mid);
        row[2 * H] = __bfloat16_as_ushort(lo);
    }
}

constexpr int kRtBN = 128;     // tokens per tile
constexpr int kRtStages = 3;
constexpr int kRtSplit = kRouterSplit;   // halves of H in separate CTAs; the top-k kernel adds the partial scores

struct RouterTcArgs {
    const float* bias;
    float* logits;   // [kRtSplit][T][E] partial scores (the bias goes into the first)
    int T, H, E;
    int32_t* hist;   // the grouping's histogram, zeroed here before the top-k kernel counts (or NULL)
    int hist_n;      // its ints
    unsigned int* status;
};

// One CTA: 128 experts x 128 tokens over one half of H, in 64-column steps.  A
// step brings the tile of x once and the hi, mid and lo tiles of W_r for the same
// columns; the three terms go into three TMEM accumulators (3 x 128 columns).
// Warp 0 issues TMA, warp 1 owns TMEM and issues the MMAs (warp-uniform, one
// elected lane), warps 4-7 write the scores.
__global__ void __launch_bounds__(256, 1)
router_tc_kernel(const __grid_constant__ RouterTcArgs a, const __grid_constant__ CUtensorMap mapA,
                 const __grid_constant__ CUtensorMap mapX) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr uint32_t TILE = kBM * kBK * 2;            // 16 KB: 128 rows x 64 bf16
    static_assert(kRtBN * kBK * 2 == TILE, "x and W_r tiles have the same size");
    constexpr uint32_t STAGE = 4 * TILE;                // x, then W_r hi, mid, lo
    uint64_t* full = reinterpret_cast<uint64_t*>(base + kRtStages * STAGE);
    uint64_t* empty = full + kRtStages;
    uint64_t* accum = empty + kRtStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(accum + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1) + 1;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kRtBN, kh = blockIdx.z;
    griddep_wait();               // programmatic dependent launch: nothing is touched before the
    griddep_launch_dependents();  // previous kernel has completed; the next one may be scheduled
    if (a.hist) {   // every CTA zeroes its share of the histogram
        const int nblk = gridDim.x * gridDim.y * gridDim.z;
        const int b = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        for (int i = b * blockDim.x + tid; i < a.hist_n; i += nblk * blockDim.x) a.hist[i] = 0;
    }
    const int hsteps = a.H / kBK, s0 = kh * hsteps / kRtSplit, s1 = (kh + 1) * hsteps / kRtSplit, nS = s1 - s0;
    if (tid == 0) {
        for (int s = 0; s < kRtStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(accum, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);   // hi, mid, lo accumulators at 0, 128, 256
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *tmem_slot;
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&mapA);
        prefetch_tensormap(&mapX);
        for (int i = 0; i < nS; ++i) {
            const int s = i % kRtStages, c = (s0 + i) * kBK;
            if (!mbar_wait(&empty[s], ((i / kRtStages) & 1) ^ 1, abort_flag, a.status)) break;
            uint8_t* st = base + (size_t)s * STAGE;
            mbar_arrive_expect_tx(&full[s], STAGE);
            tma_load_2d(st, &mapX, c, n0, &full[s]);
            for (int part = 0; part < 3; ++part) tma_load_2d(st + (1 + part) * TILE, &mapA, part * a.H + c, m0, &full[s]);
        }
    } else if (warp == 1) {   // warp-uniform loop, one elected lane issues
        const uint32_t idesc = umma_idesc_bf16(kBM, kRtBN);
        bool ok = true;
        for (int i = 0; i < nS; ++i) {
            const int s = i % kRtStages;
            if (!(ok = mbar_wait_warp(&full[s], (i / kRtStages) & 1, abort_flag, a.status))) break;
            tc_fence_after();
            const uint32_t sb = smem_u32(base + (size_t)s * STAGE);
            const uint64_t bdesc0 = umma_desc_sw128(sb);
            // one accumulator per term: products of very different magnitude are
            // never summed inside the tensor core, only in fp32 in the epilogue
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                const uint64_t adesc0 = umma_desc_sw128(sb + (1 + part) * TILE);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)   // +32 bytes per K=16 slice: +2 in the address field
                    umma_f16_elect(taddr + part * kRtBN, adesc0 + 2 * kk, bdesc0 + 2 * kk, idesc, (i | kk) != 0);
            }
            umma_commit_elect(&empty[s]);
        }
        if (ok) umma_commit_elect(accum);
    } else if (warp >= 4) {
        const int q = warp - 4, e = m0 + q * 32 + lane;
        if (mbar_wait(accum, 0, abort_flag, a.status)) {
            tc_fence_after();
            const float bias = (kh == 0 && e < a.E && a.bias) ? a.bias[e] : 0.f;
            float* out = a.logits + (size_t)kh * a.T * a.E;
            for (int c0 = 0; c0 < kRtBN; c0 += 16) {
                uint32_t vh[16], vm[16], vl[16];
                const uint32_t ta = taddr + ((uint32_t)(q * 32) << 16) + c0;
                tmem_ld16(ta, vh);
                tmem_ld16(ta + kRtBN, vm);
                tmem_ld16(ta + 2 * kRtBN, vl);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = n0 + c0 + j;
                    const float v = __uint_as_float(vh[j]) + (__uint_as_float(vm[j]) + __uint_as_float(vl[j]));
                    if (e < a.E && t < a.T) out[(size_t)t * a.E + e] = v + bias;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(taddr, 512);
}

size_t router_tc_smem() { return 1024 + (size_t)kRtStages * 4 * kBM * kBK * 2 + 2 * kRtStages * 8 + 32; }

// ---------------------------------------------------------------------------
// per-token selection: one warp per token
// ---------------------------------------------------------------------------
constexpr int kTopkWarps = 8;

// NIT >= ceil(H/256): 16-byte loads of the x row per lane, held in registers.
template <int NIT>
__global__ void __launch_bounds__(kTopkWarps * 32, NIT <= 8 ? 4 : 2) topk_kernel(const float* __restrict__ logits,
                                                               int nsplit,   // 1 or 2 partial score arrays
                                                               const uint16_t* __restrict__ x,
                                                               const float* __restrict__ g, int T, int H, int E,
                                                               int k, int32_t* __restrict__ idx,
                                                               float* __restrict__ w, float* __restrict__ gamma,
                                                               uint16_t* __restrict__ x16, int bits,
                                                               int32_t* __restrict__ hist, unsigned int* status) {
    extern __shared__ float sm_topk[];
    float* gs = sm_topk;                    // [H] shared-expert gate vector, staged once per block
    float* sc_all = sm_topk + H;            // [kTopkWarps][E] scores
    uint16_t* xs_all = reinterpret_cast<uint16_t*>(sc_all + kTopkWarps * E);   // [kTopkWarps][H] rows of x
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    griddep_wait();               // programmatic dependent launch: nothing is touched before the
    griddep_launch_dependents();  // previous kernel has completed; the next one may be scheduled
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x)
        reinterpret_cast<float4*>(gs)[i] = reinterpret_cast<const float4*>(g)[i];
    __syncthreads();
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    // the token's row of x is requested first, into shared memory (no registers held
    // across the selection), so that its latency hides behind the selection
    uint16_t* xs = xs_all + (size_t)warp * H;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int h = it * 256 + lane * 8;
        if (h < H) cp_async_16(xs + h, x + (size_t)t * H + h);
    }
    cp_async_commit();
    float* sc = sc_all + warp * E;
    // partial scores added in order; unrolled so that the loads of a row are in flight together
    const float* l0 = logits + (size_t)t * E;
    const float* l1 = logits + ((size_t)T + t) * E;
#pragma unroll 8
    for (int e = lane; e < E; e += 32) sc[e] = nsplit > 1 ? l0[e] + l1[e] : l0[e];
    __syncwarp();
    select_topk_warp(sc, E, k, idx + (size_t)t * k, w + (size_t)t * k);
    // the grouping's histogram: assignments per (chunk of kChunk tokens, expert)
    // (each lane reads back the selection it wrote)
    if (hist && lane < k) atomicAdd(&hist[(size_t)(t / kChunk) * E + idx[(size_t)t * k + lane]], 1);
    float d = 0.f;
    bool fits = true;
    cp_async_wait<0>();   // each lane reads back only the chunks it copied
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int h = it * 256 + lane * 8;
        if (h >= H) break;
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + h);
        const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
        const float4 g0 = *reinterpret_cast<const float4*>(gs + h), g1 = *reinterpret_cast<const float4*>(gs + h + 4);
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(u[i] << 16);
            f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            d = fmaf(f[i], gg[i], d);
            fits = fits && fabsf(f[i]) <= 65504.f;
        }
        // fp16 copy in the K order the dequantised weights use: 4-bit codes
        // {0,4,1,5,2,6,3,7}, 8-bit codes {0,2,1,3,4,6,5,7} per 8 columns
        if (x16) {
            uint32_t hv[4];
            if (bits == 8) {
                hv[0] = h2_as_u32(__floats2half2_rn(f[0], f[2]));
                hv[1] = h2_as_u32(__floats2half2_rn(f[1], f[3]));
                hv[2] = h2_as_u32(__floats2half2_rn(f[4], f[6]));
                hv[3] = h2_as_u32(__floats2half2_rn(f[5], f[7]));
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) hv[i] = h2_as_u32(__floats2half2_rn(f[i], f[i + 4]));
            }
            *reinterpret_cast<uint4*>(x16 + (size_t)t * H + h) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        }
    }
    if (x16 && !fits) raise_status(status, MOE_W4_STATUS_FP16_RANGE);
    d = warp_sum(d);
    if (lane == 0) gamma[t] = 1.0f / (1.0f + expf(-d));
}

typedef CUresult (*EncodeTiledFnR)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static bool bf16_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    static EncodeTiledFnR fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<EncodeTiledFnR>(p);
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Dynamic shared memory of topk_kernel: the gate vector, the warps' scores and
// the warps' rows of x; largest for H = 4096, E = 1024.
static size_t topk_smem(int H, int E) {
    return ((size_t)H + (size_t)kTopkWarps * E) * sizeof(float) + (size_t)kTopkWarps * H * 2;
}
static cudaError_t topk_smem_attr() {
    static bool done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    const int mx = (int)topk_smem(4096, 1024);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(topk_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

size_t router_prep_bytes(const moe_w4_layer& L) {
    const size_t Epad = (size_t)(L.E + kBM - 1) / kBM * kBM;
    return Epad * 3 * (size_t)L.H * 2;
}

cudaError_t launch_router_prep(const moe_w4_layer& L, uint16_t* dst, cudaStream_t st) {
    const int Epad = (L.E + kBM - 1) / kBM * kBM;
    router_split_kernel<<<dim3(L.H / 32, Epad / 32), 256, 0, st>>>(L.router_w, L.H, L.E, Epad, dst);
    return cudaGetLastError();
}

cudaError_t launch_router_prefill(const moe_w4_layer& L, int T, const uint16_t* x, const RouteOut& o,
                                  cudaStream_t st) {
    const int Epad = (L.E + kBM - 1) / kBM * kBM;
    {
        const cudaError_t e = topk_smem_attr();
        if (e != cudaSuccess) return e;
    }
    // the split router weights: prepared once per layer (moe_w4_prepare_router),
    // else split into the workspace on every call
    const uint16_t* ra = static_cast<const uint16_t*>(L.router_prep);
    if (!ra) {
        router_split_kernel<<<dim3(L.H / 32, Epad / 32), 256, 0, st>>>(L.router_w, L.H, L.E, Epad, o.router_a);
        ra = o.router_a;
    }
    {
        CUtensorMap mA, mX;
        if (!bf16_map(&mA, ra, Epad, 3 * (uint64_t)L.H, kBM) || !bf16_map(&mX, x, T, L.H, kRtBN))
            return cudaErrorInvalidValue;
        static size_t attr[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (attr[dev] < router_tc_smem()) {
            const cudaError_t e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)router_tc_smem());
            if (e != cudaSuccess) return e;
            attr[dev] = router_tc_smem();
        }
        // the grouping's per-chunk histogram, zeroed by this kernel, counted by the top-k kernel
        RouterTcArgs ra_args{L.router_bias, o.logits, T, L.H, L.E, o.chunk_base,
                             ((T + kChunk - 1) / kChunk) * L.E, o.status};
        const cudaError_t e = launch_pdl(pdl_for(T), router_tc_kernel, dim3(Epad / kBM, (T + kRtBN - 1) / kRtBN, kRtSplit),
                                         dim3(256), router_tc_smem(), st, ra_args, mA, mX);
        if (e != cudaSuccess) return e;
    }
    trace_mark(st, 1);
    const int nsplit = kRtSplit;
    const size_t sm = topk_smem(L.H, L.E);
    const dim3 grid((T + kTopkWarps - 1) / kTopkWarps), block(kTopkWarps * 32);
    const int nit = (L.H + 255) / 256;   // H <= 4096
    auto topk = nit <= 2 ? topk_kernel<2> : nit <= 4 ? topk_kernel<4> : nit <= 8 ? topk_kernel<8> : topk_kernel<16>;
    const cudaError_t e = launch_pdl(pdl_for(T), topk, grid, block, sm, st, o.logits, nsplit, x, L.shared_gate, T, L.H, L.E,
                                     L.top_k, o.topk_idx, o.topk_w, o.gamma, o.x16, code_bits_of(L), o.chunk_base,
                                     o.status);
    if (e != cudaSuccess) return e;
    trace_mark(st, 2);
    return cudaGetLastError();
}

}  // namespace mw4
