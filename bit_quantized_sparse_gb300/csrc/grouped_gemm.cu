// Prefill expert FFN as grouped GEMMs on the 5th-generation tensor cores.
// Operands are fp16 (weights rebuilt in fp16, activations and the intermediate
// h in fp16), accumulation fp32: fp16 has the same tcgen05 rate as bf16 and
// eight times its precision, which keeps the computation error an order of
// magnitude below the rounding of the bf16 output.
// ("Optimizing on-device inference for Apple Silicon", section "Dequantise
// weights during matrix multiplication": the tensor operations want bf16
// operands, so each small weight tile is rebuilt in bf16 in on-chip memory
// just before it multiplies the routed activation rows; accumulation is fp32,
// output bf16, and the expanded weight array never exists in memory.  Section
// "Match tile size to expert load": tiles of fixed size over each expert's
// rows, listed in a block map.)
//
// One CTA computes one tile: 128 weight rows (output features) x up to 128
// grouped token rows, reducing over K in 64-column steps (one quantisation
// group per row per step).  Warp roles, 384 threads:
//   warp 0      TMA: packed codes of the step (and, for the down projection,
//               the activation rows), plus the tile's scales/biases once
//   warp 1      TMEM allocation; one thread issues tcgen05.mma
//   warps 2-3   gate/up only: gather the token rows of x with cp.async
//   warps 4-11  dequantise codes -> bf16 A tiles (128-byte swizzle) in smem;
//               warps 4-7 then run the epilogue out of TMEM
// The weights are the M=128 operand ("swap AB"), so an expert with few rows
// wastes only N columns, and N = rows rounded up to 16.
//   gate/up:  D_g = Wg * X^T, D_u = Wu * X^T (two accumulators), epilogue
//             h = silu(D_g) * D_u -> hh[p][i] fp16
//   down:     D = Wd * H^T, epilogue scales column p by its routing weight
//             (or the shared gate) -> ys[p][o] fp16
// combine_kernel then sums, per token, its k rows of ys and the shared row in
// a fixed order.
#include "common.cuh"
#include "internal.h"

namespace mw4 {

struct GemmArgs {
    const Tile* tiles;
    const int32_t* ntiles;     // tile count (device)
    const int32_t* offsets;    // expert group starts
    const int32_t* perm;       // grouped position -> t*k + j
    const uint16_t* x16;       // [T][H] fp16 copy of the activations (gate/up)
    const float* topk_w;       // [T*k] (down)
    const float* gamma;        // [T] (down)
    const uint16_t* s0r; const uint16_t* b0r; const uint16_t* s1r; const uint16_t* b1r;   // routed
    const uint16_t* s0s; const uint16_t* b0s; const uint16_t* s1s; const uint16_t* b1s;   // shared
    const uint32_t* c0r; const uint32_t* c1r; const uint32_t* c0s; const uint32_t* c1s;   // codes (L2 prefetch)
    uint16_t* out;             // hh [.][I] or ys [.][H]
    const uint16_t* hh_rows;   // down: the B rows (hh), for the L2 prefetch
    int E, k, T, H;            // H: row length of x
    int K;                     // reduction length (H or I)
    int rows_e;                // weight rows per expert (I or H)
    int out_cols;              // I or H
    int stages;
    unsigned int* status;
};

constexpr int kThreads = 384;
constexpr uint32_t kCodesBytes = kBM * (kBK / 8) * 4;   // 4 KB of packed codes per matrix per step
constexpr uint32_t kTileBytes = kBM * kBK * 2;          // 16 KB bf16 tile (A or B)

template <bool DUAL>
struct Smem {
    static constexpr int NMAT = DUAL ? 2 : 1;
    static constexpr uint32_t stage_bytes = NMAT * kTileBytes + kTileBytes + NMAT * kCodesBytes;
    static size_t bytes(int stages, int K) {
        const size_t sb = (size_t)NMAT * 2 * kBM * (K / kGroup) * 2;
        return 1024 + (size_t)stages * stage_bytes + sb + (4 * stages + 2) * 8 + 16 + kBN * 4;
    }
};

MW4_DEV uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <bool DUAL>
__global__ void __launch_bounds__(kThreads, 1)
grouped_w4_gemm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap map0r,
                       const __grid_constant__ CUtensorMap map1r, const __grid_constant__ CUtensorMap map0s,
                       const __grid_constant__ CUtensorMap map1s, const __grid_constant__ CUtensorMap mapb) {
    constexpr int NMAT = Smem<DUAL>::NMAT;
    constexpr uint32_t NCOLS = DUAL ? 256 : 128;
    if ((int)blockIdx.x >= a.ntiles[0]) return;
    const Tile tile = a.tiles[blockIdx.x];
    const int S = a.stages, G = a.K / kGroup, nK = a.K / kBK;
    const bool shared_e = (tile.e == a.E);
    const int p0 = (shared_e ? a.T * a.k : a.offsets[tile.e]) + tile.r0;
    const int arow = (shared_e ? 0 : tile.e * a.rows_e) + tile.m * kBM;
    const int nrows = tile.nrows;
    const int nmma = ((nrows + 15) / 16) * 16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align1024(smem_raw);
    auto A_of = [&](int s, int mat) { return base + (size_t)s * Smem<DUAL>::stage_bytes + mat * kTileBytes; };
    auto B_of = [&](int s) { return base + (size_t)s * Smem<DUAL>::stage_bytes + NMAT * kTileBytes; };
    auto C_of = [&](int s, int mat) {
        return reinterpret_cast<uint32_t*>(base + (size_t)s * Smem<DUAL>::stage_bytes + (NMAT + 1) * kTileBytes +
                                           mat * kCodesBytes);
    };
    uint16_t* sb = reinterpret_cast<uint16_t*>(base + (size_t)S * Smem<DUAL>::stage_bytes);   // [NMAT][2][128][G]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb + (size_t)NMAT * 2 * kBM * G);
    uint64_t* full_codes = bars;
    uint64_t* full_B = bars + S;
    uint64_t* full_A = bars + 2 * S;
    uint64_t* empty = bars + 3 * S;
    uint64_t* sb_full = bars + 4 * S;
    uint64_t* accum_full = bars + 4 * S + 1;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 4 * S + 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4 * S + 2) + 1;
    float* col_scale = reinterpret_cast<float*>(bars + 4 * S + 2) + 4;   // [kBN], 16-byte aligned

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_codes[s], 1);
            mbar_init(&full_B[s], 64);
            mbar_init(&full_A[s], 256);
            mbar_init(&empty[s], 1);
        }
        mbar_init(sb_full, 1);
        mbar_init(accum_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, NCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const CUtensorMap* m0 = shared_e ? &map0s : &map0r;
            const CUtensorMap* m1 = shared_e ? &map1s : &map1r;
            prefetch_tensormap(m0);
            if (DUAL) prefetch_tensormap(m1); else prefetch_tensormap(&mapb);
            // the tile's packed codes are one contiguous range per matrix: pull
            // them into L2 now so the per-step TMA loads hit L2, not HBM
            const size_t coff = (size_t)arow * (a.K / 8);
            const uint32_t cbytes = kBM * (a.K / 2);
            prefetch_l2((shared_e ? a.c0s : a.c0r) + coff, cbytes);
            if (DUAL) prefetch_l2((shared_e ? a.c1s : a.c1r) + coff, cbytes);
            else prefetch_l2(a.hh_rows + (size_t)p0 * a.K, (uint32_t)nrows * a.K * 2);
            const size_t goff = shared_e ? (size_t)tile.m * kBM * G : ((size_t)tile.e * a.rows_e + tile.m * kBM) * G;
            const uint32_t sbb = kBM * G * 2;
            mbar_arrive_expect_tx(sb_full, NMAT * 2 * sbb);
            bulk_load(sb, (shared_e ? a.s0s : a.s0r) + goff, sbb, sb_full);
            bulk_load(sb + kBM * G, (shared_e ? a.b0s : a.b0r) + goff, sbb, sb_full);
            if (DUAL) {
                bulk_load(sb + 2 * kBM * G, (shared_e ? a.s1s : a.s1r) + goff, sbb, sb_full);
                bulk_load(sb + 3 * kBM * G, (shared_e ? a.b1s : a.b1r) + goff, sbb, sb_full);
            }
            for (int ks = 0; ks < nK; ++ks) {
                const int s = ks % S;
                const uint32_t ph = (ks / S) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, a.status)) break;
                mbar_arrive_expect_tx(&full_codes[s], NMAT * kCodesBytes + (DUAL ? 0 : kTileBytes));
                tma_load_2d(C_of(s, 0), m0, ks * (kBK / 8), arow, &full_codes[s]);
                if (DUAL) tma_load_2d(C_of(s, 1), m1, ks * (kBK / 8), arow, &full_codes[s]);
                else tma_load_2d(B_of(s), &mapb, ks * kBK, p0, &full_codes[s]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16(kBM, nmma);
            bool ok = true;
            for (int ks = 0; ks < nK && ok; ++ks) {
                const int s = ks % S;
                const uint32_t ph = (ks / S) & 1;
                ok = mbar_wait(&full_A[s], ph, abort_flag, a.status) &&
                     mbar_wait(DUAL ? &full_B[s] : &full_codes[s], ph, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t bdesc = umma_desc_sw128(smem_u32(B_of(s)) + kk * 32);
#pragma unroll
                    for (int mat = 0; mat < NMAT; ++mat) {
                        const uint64_t adesc = umma_desc_sw128(smem_u32(A_of(s, mat)) + kk * 32);
                        umma_f16(taddr + mat * 128, adesc, bdesc, idesc, (ks | kk) != 0);
                    }
                }
                umma_commit(&empty[s]);
            }
            if (ok) umma_commit(accum_full);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ token-row gather (gate/up)
        if (DUAL) {
            const int tb = tid - 64, c = tb & 7;
            int tok[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int row = (tb >> 3) + 8 * n;
                tok[n] = -1;
                if (row < nrows) tok[n] = shared_e ? tile.r0 + row : a.perm[p0 + row] / a.k;
            }
            // up to `lag` gathers stay in flight; stage ks is signalled once its
            // own copies have landed (cp.async.wait_group), after a proxy fence
            const int lag = S - 1 < 2 ? S - 1 : 2;
            bool ok = true;
            int signalled = 0;
            for (int ks = 0; ks < nK; ++ks) {
                const int s = ks % S;
                const uint32_t ph = (ks / S) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, a.status)) { ok = false; break; }
                uint8_t* dst = B_of(s);
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const int row = (tb >> 3) + 8 * n;
                    if (tok[n] >= 0)
                        cp_async_16(dst + row * 128 + ((c ^ (row & 7)) << 4),
                                    a.x16 + (size_t)tok[n] * a.H + ks * kBK + c * 8);
                }
                cp_async_commit();
                if (ks - signalled >= lag) {
                    if (lag == 2) cp_async_wait<2>(); else cp_async_wait<1>();
                    fence_proxy_async_smem();
                    mbar_arrive(&full_B[signalled % S]);
                    ++signalled;
                }
            }
            cp_async_wait<0>();
            if (ok) {
                fence_proxy_async_smem();
                for (; signalled < nK; ++signalled) mbar_arrive(&full_B[signalled % S]);
            }
        }
    } else {
        // ------------------------------------------------------------ dequantisation
        const int td = tid - 128, word = td & 7, rbase = td >> 3;
        bool ok = mbar_wait(sb_full, 0, abort_flag, a.status);
        // scales and biases arrive as bf16; convert the tile to fp16 once (exact
        // for normal values), shared by the 256 dequantising threads
        uint16_t* sb16 = sb;
        for (int i = td; i < NMAT * 2 * kBM * G && ok; i += 256)
            sb16[i] = __half_as_ushort(__float2half_rn(bf16_bits_to_float(sb[i])));
        asm volatile("bar.sync 1, 256;" ::: "memory");
        for (int ks = 0; ks < nK && ok; ++ks) {
            const int s = ks % S;
            const uint32_t ph = (ks / S) & 1;
            if (!mbar_wait(&full_codes[s], ph, abort_flag, a.status)) { ok = false; break; }
#pragma unroll
            for (int mat = 0; mat < NMAT; ++mat) {
                const uint32_t* cw = C_of(s, mat);
                uint8_t* At = A_of(s, mat);
                const uint16_t* ss = sb16 + (size_t)(2 * mat) * kBM * G;
                const uint16_t* bb = ss + (size_t)kBM * G;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = rbase + 32 * j;
                    const uint32_t w = cw[row * 8 + word];
                    const uint32_t s16 = ss[row * G + ks], b16 = bb[row * G + ks];
                    uint32_t o[4];
                    dequant8_f16(w, u32_as_h2(s16 | (s16 << 16)), u32_as_h2(b16 | (b16 << 16)), o);
                    *reinterpret_cast<uint4*>(At + row * 128 + ((word ^ (row & 7)) << 4)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&full_A[s]);
        }
        // ------------------------------------------------------------ epilogue (warps 4-7)
        if (!DUAL && warp < 8) {   // per-column output scale, fetched while the MMAs run
            const int i = tid - 128;
            if (i < nrows) col_scale[i] = shared_e ? a.gamma[tile.r0 + i] : a.topk_w[a.perm[p0 + i]];
            asm volatile("bar.sync 2, 128;" ::: "memory");
        }
        if (warp < 8 && ok && mbar_wait(accum_full, 0, abort_flag, a.status)) {
            tc_fence_after();
            const int q = warp - 4;
            const uint32_t lane_addr = taddr + ((uint32_t)(q * 32) << 16);
            const int ocol = tile.m * kBM + q * 32 + lane;
            for (int c0 = 0; c0 < nrows; c0 += 16) {
                uint32_t g[16], u[16];
                tmem_ld16(lane_addr + c0, g);
                if (DUAL) tmem_ld16(lane_addr + 128 + c0, u);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c0 + j;
                    if (n >= nrows) break;
                    float v;
                    if (DUAL) {
                        v = silu_f(__uint_as_float(g[j])) * __uint_as_float(u[j]);
                    } else {
                        v = __uint_as_float(g[j]) * col_scale[n];
                    }
                    if (!(fabsf(v) <= 65504.f)) raise_status(a.status, MOE_W4_STATUS_FP16_RANGE);
                    a.out[(size_t)(p0 + n) * a.out_cols + ocol] = __half_as_ushort(__float2half_rn(v));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(taddr, NCOLS);
}

// out[t] = bf16( sum_j ys[inv[t*k + j]] + ys[T*k + t] ) with ys in fp16 and
// the sum in fp32, slots in order then the shared row; 8 columns per thread.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ ys,
                                                      const int32_t* __restrict__ inv, uint16_t* __restrict__ out,
                                                      int T, int H, int k) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int per_row = H / 8;
    if (i >= (size_t)T * per_row) return;
    const int t = (int)(i / per_row), c = (int)(i % per_row) * 8;
    float acc[8] = {};
    for (int j = 0; j <= k; ++j) {
        const size_t p = (j < k) ? (size_t)inv[(size_t)t * k + j] : (size_t)T * k + t;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(ys + p * H + c));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(u32_as_h2(u[q]));
            acc[2 * q] += f.x;
            acc[2 * q + 1] += f.y;
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        o[q] = bf162_as_u32(__floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]));
    *reinterpret_cast<uint4*>(out + (size_t)t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2D map over a row-major [rows][cols] tensor, box [box_rows][box_cols].
static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* ptr, uint64_t rows,
                     uint64_t cols, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int stages_for(bool dual, int K) {
    const int budget = 227 * 1024;
    for (int s = 4; s >= 2; --s) {
        const size_t b = dual ? Smem<true>::bytes(s, K) : Smem<false>::bytes(s, K);
        if (b <= (size_t)budget) return s;
    }
    return 0;
}

cudaError_t launch_grouped_ffn(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out, const PrefillWs& p,
                               cudaStream_t st) {
    const int H = L.H, I = L.I, E = L.E, k = L.top_k;
    const uint64_t rows_all = (uint64_t)T * k + T;
    CUtensorMap mg, mu, msg, msu, md, msd, mh;
    const auto U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32;
    bool ok = make_map(&mg, U32, 4, L.gate.codes, (uint64_t)E * I, H / 8, kBM, kBK / 8, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&mu, U32, 4, L.up.codes, (uint64_t)E * I, H / 8, kBM, kBK / 8, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&msg, U32, 4, L.sh_gate.codes, I, H / 8, kBM, kBK / 8, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&msu, U32, 4, L.sh_up.codes, I, H / 8, kBM, kBK / 8, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&md, U32, 4, L.down.codes, (uint64_t)E * H, I / 8, kBM, kBK / 8, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&msd, U32, 4, L.sh_down.codes, H, I / 8, kBM, kBK / 8, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&mh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.hh, rows_all, I, kBN, kBK,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;

    const int s_gu = stages_for(true, H), s_dn = stages_for(false, I);
    if (s_gu == 0 || s_dn == 0) return cudaErrorInvalidConfiguration;
    const size_t sm_gu = Smem<true>::bytes(s_gu, H), sm_dn = Smem<false>::bytes(s_dn, I);
    static int set_gu[64] = {}, set_dn[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (set_gu[dev] < (int)sm_gu) {
        cudaFuncSetAttribute(grouped_w4_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_gu);
        set_gu[dev] = (int)sm_gu;
    }
    if (set_dn[dev] < (int)sm_dn) {
        cudaFuncSetAttribute(grouped_w4_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_dn);
        set_dn[dev] = (int)sm_dn;
    }

    GemmArgs a{};
    a.ntiles = p.ntiles; a.offsets = p.offsets; a.perm = p.perm; a.x16 = p.x16;
    a.topk_w = p.topk_w; a.gamma = p.gamma;
    a.E = E; a.k = k; a.T = T; a.H = H; a.status = p.status;

    // gate/up: A = Wg, Wu rows (I per expert), K = H, out = hh [.][I]
    a.tiles = p.tiles_gu;
    a.s0r = L.gate.scales; a.b0r = L.gate.biases; a.s1r = L.up.scales; a.b1r = L.up.biases;
    a.s0s = L.sh_gate.scales; a.b0s = L.sh_gate.biases; a.s1s = L.sh_up.scales; a.b1s = L.sh_up.biases;
    a.c0r = L.gate.codes; a.c1r = L.up.codes; a.c0s = L.sh_gate.codes; a.c1s = L.sh_up.codes;
    a.out = p.hh; a.K = H; a.rows_e = I; a.out_cols = I; a.stages = s_gu;
    grouped_w4_gemm_kernel<true><<<p.max_tiles_gu, kThreads, sm_gu, st>>>(a, mg, mu, msg, msu, mh);
    trace_mark(st, 6);

    // down: A = Wd rows (H per expert), K = I, B = hh rows, out = ys [.][H]
    GemmArgs b = a;
    b.tiles = p.tiles_dn; b.ntiles = p.ntiles + 1;
    b.s0r = L.down.scales; b.b0r = L.down.biases; b.s1r = nullptr; b.b1r = nullptr;
    b.s0s = L.sh_down.scales; b.b0s = L.sh_down.biases; b.s1s = nullptr; b.b1s = nullptr;
    b.c0r = L.down.codes; b.c1r = nullptr; b.c0s = L.sh_down.codes; b.c1s = nullptr; b.hh_rows = p.hh;
    b.out = p.ys; b.K = I; b.rows_e = H; b.out_cols = H; b.stages = s_dn;
    grouped_w4_gemm_kernel<false><<<p.max_tiles_dn, kThreads, sm_dn, st>>>(b, md, md, msd, msd, mh);
    trace_mark(st, 7);

    const size_t nthr = (size_t)T * (H / 8);
    combine_kernel<<<(unsigned)((nthr + 255) / 256), 256, 0, st>>>(p.ys, p.inv, out, T, H, k);
    trace_mark(st, 8);
    return cudaGetLastError();
}

}  // namespace mw4
