// Prefill expert FFN as grouped GEMMs on the 5th-generation tensor cores.
// Along K every operand is stored in chunk order (common.cuh): the
// dequantised weights come out that way, the fp16 copy of x and h are written
// that way.
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
// A tile is 128 weight rows (output features) x up to 128 grouped token rows,
// reduced over K in 128-column steps (two quantisation groups per row per step).
// The weights are the M=128 operand ("swap AB"), so an expert with few rows
// wastes only N columns, and N = rows rounded up to 16.
//   gate/up:  D_g = Wg * X^T, D_u = Wu * X^T (two accumulators), epilogue
//             h = w_p * silu(D_g) * D_u -> hh[p][i] fp16, w_p the routing weight
//             of grouped row p (or the shared gate): the down projection is
//             linear, so weighting its input weights its output
//   down:     D = Wd * H^T -> ys[p][o] fp16
// The kernel is persistent (one CTA per SM, tiles strided by the grid) and
// warp-specialised:
//   dequantisers  8 warps (gate/up: one thread per matrix row; down: two threads
//                 per row, one group of the step each): codes from
//                 shared memory -> fp16 -> tcgen05.st into an A ring in TMEM
//   epilogue      8 warps, two per TMEM lane quarter: TMEM -> registers ->
//                 global memory
//   producer      1 warp, TMA: the step's packed codes and the tile's B rows,
//                 contiguous in grouped order (gate/up: the token rows copied
//                 by gather_rows_kernel, or x16 itself for the shared expert;
//                 down: hh); no L2 prefetch of codes or rows (measured slower: the
//                 prefetches occupy the TMA unit at every tile start)
//   MMA           1 warp: TMEM allocation and the MMA loop (warp-uniform, one
//                 elected lane issues tcgen05.mma with A read from tensor memory)
// gather_rows_kernel first copies the token rows of x16 into grouped order, so
// that every B row block is one contiguous range for TMA.
// combine_kernel then sums, per token, its k rows of ys and the shared row in
// a fixed order.
#include "common.cuh"
#include "internal.h"

namespace mw4 {

struct GemmArgs {
    const int4* blkinfo;       // per 128-row block: {group (E = shared), first row, rows, first grouped position}
    const int4* unitinfo;      // down: units {first row block, row blocks, group, 0}; NULL: one block per unit
    const int32_t* ntiles;     // tile count (device)
    int M;                     // weight-row blocks (work item = unit * M + weight-row block)
    const int32_t* offsets;    // expert group starts
    const int32_t* perm;       // grouped position -> t*k + j
    const float* topk_w;       // [T*k] (gate/up epilogue)
    const float* gamma;        // [T] (gate/up epilogue)
    const uint16_t* s0r; const uint16_t* b0r; const uint16_t* s1r; const uint16_t* b1r;   // routed
    const uint16_t* s0s; const uint16_t* b0s; const uint16_t* s1s; const uint16_t* b1s;   // shared
    uint16_t* out;             // hh [.][I] or ys [.][H]
    int E, k, T, H;            // H: row length of x
    int K;                     // reduction length (H or I)
    int rows_e;                // weight rows per expert (I or H)
    int out_cols;              // I or H
    int k_order8;              // K order of the one-byte codes (fp16 weights from a separate pass only)
    int max_blocks;            // capacity of the block (and unit) records (debug-build bounds)
    unsigned int* status;
};

constexpr int kGK = 128;                                // reduction columns per pipeline step
static_assert(kGK == 2 * kGroup, "a step holds two quantisation groups");
constexpr uint32_t kSubBytes = kBN * 64 * 2;            // 16 KB: 128 B rows x 64 fp16 columns, 128-byte swizzle
constexpr uint32_t kTileBytes = 2 * kSubBytes;          // B tile of one step: two K sub-tiles

// Persistent-kernel geometry: warp roles, ring depths and the TMEM map.
// The dequantised weights (the A operand) live in tensor memory, written by
// tcgen05.st and read by the MMA from there: no shared-memory round trip and
// no proxy fence.  TMEM (512 columns) holds the accumulators and an A ring.
template <bool DUAL, int BITS>
struct Geo {
    static constexpr int NMAT = DUAL ? 2 : 1;
    // packed codes of one weight row per step (64 B for 4-bit, 128 B for 8-bit codes)
    static constexpr uint32_t kCodesRowBytes = kGK * BITS / 8;
    static constexpr uint32_t kCodesBytes = kBM * kCodesRowBytes;   // per matrix per step
    // 8 dequantiser warps: gate/up one thread per (matrix, weight row); down two
    // threads per weight row, one of the step's two groups each (more threads in
    // flight for the one matrix)
    static constexpr int kDeqWarps = 8;
    static constexpr int kDeqWarp0 = 0;                   // warp w reaches TMEM lanes 32*(w%4)..+31, so the
    static constexpr int kEpiWarp0 = kDeqWarp0 + kDeqWarps;   // dequantiser and epilogue groups start at w%4 == 0
    static constexpr int kEpiWarps = 8;                   // two per TMEM lane group, columns interleaved
    static constexpr int kProdWarp = kEpiWarp0 + kEpiWarps;   // TMA producer of the codes
    static constexpr int kProdBWarp = kProdWarp + 1;          // TMA producer of the B rows
    static constexpr int kMmaWarp = kProdBWarp + 1;           // TMEM owner and MMA issuer
    static constexpr int kThreads = 32 * (kMmaWarp + 1);
    // Two rings in shared memory: the codes, freed as soon as the dequantisers
    // have read a step, and the B rows, freed when the step's MMAs complete.
    // The codes thus run several steps ahead of the dequantisers, whatever the
    // MMAs' lag.
    // BITS = 16: weights already rebuilt in fp16 by a separate pass (a
    // measurement-only variant): the "codes" ring holds fp16 A tiles that the
    // MMAs read from shared memory, and no dequantiser runs
    static constexpr int SC = BITS == 16 ? (DUAL ? 2 : 3) : DUAL ? (BITS == 8 ? 3 : 4) : (BITS == 8 ? 6 : 8);
    static constexpr int SB = BITS == 16 ? (DUAL ? 2 : 3) : 4;
    static constexpr uint32_t C_STAGE = NMAT * kCodesBytes;
    static constexpr uint32_t ACC_COLS = NMAT * 128;      // TMEM columns per accumulator buffer
    static constexpr int ACC_BUFS = DUAL ? 1 : 2;
    static constexpr uint32_t A_COLS = NMAT * (kGK / 2);  // TMEM columns per A stage (16-bit pairs)
    static constexpr int SA = (512 - ACC_BUFS * ACC_COLS) / A_COLS;   // A ring in TMEM
    static constexpr uint32_t A_TMEM0 = ACC_BUFS * ACC_COLS;
    static constexpr size_t bytes() {
        return 1024 + (size_t)SB * kTileBytes + (size_t)SC * C_STAGE + 2 * kBN * 4 +
               (2 * SB + 2 * SC + 2 * SA + 4) * 8 + 16;
    }
};
static_assert(Geo<true, 4>::SA == 2 && Geo<false, 4>::SA == 4, "TMEM map");
static_assert(Geo<true, 4>::bytes() <= 232448 && Geo<false, 4>::bytes() <= 232448, "shared memory per CTA");
static_assert(Geo<true, 8>::bytes() <= 232448 && Geo<false, 8>::bytes() <= 232448, "shared memory per CTA");
static_assert(Geo<true, 16>::bytes() <= 232448 && Geo<false, 16>::bytes() <= 232448, "shared memory per CTA");
static_assert(kDownReuseMaxI / kGK <= Geo<false, 4>::SA, "a reused down weight tile holds its whole K in the A ring");
static_assert(Geo<true, 4>::SA <= Geo<true, 4>::SB, "gate/up A slots are freed by the B-ring barriers");

MW4_DEV uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct TileInfo { int e, m, r0, nrows, p0, arow; bool sh; };
struct UnitInfo { int b0, nb, m; };

// Work item t = (unit t / M, weight-row block t % M).  A unit is a run of row
// blocks of one group (a single block unless unitinfo is given): its weight
// tile is dequantised once and multiplied with each of its row blocks.
// A unit record {first row block, row blocks} (checked in debug builds: at
// most kDownBlocksPerUnit blocks, inside the block records).
MW4_DEV int2 checked_unit(const GemmArgs& a, int b0, int nb) {
    nb = checked_index(nb, 1, kDownBlocksPerUnit + 1, a.status);
    b0 = checked_index(b0, 0, a.max_blocks - nb + 1, a.status);
    return make_int2(b0, nb);
}

MW4_DEV UnitInfo unit_info(const GemmArgs& a, int t) {
    UnitInfo u;
    u.m = t % a.M;
    if (a.unitinfo) {
        const int4 r = __ldg(a.unitinfo + t / a.M);
        const int2 c = checked_unit(a, r.x, r.y);
        u.b0 = c.x;
        u.nb = c.y;
    } else {
        u.b0 = t / a.M;
        u.nb = 1;
    }
    return u;
}

// Unit record of work item t as {first row block, row blocks}: no load when
// every unit is one block; {0, 0} past the last item.
MW4_DEV int2 unit_rec(const GemmArgs& a, int t, int ntiles) {
    if (t >= ntiles) return make_int2(0, 0);
    if (!a.unitinfo) return make_int2(t / a.M, 1);
    const int4 r = __ldg(a.unitinfo + t / a.M);
    return checked_unit(a, r.x, r.y);
}

// Tile (row block with record bi, weight-row block m); the record (group,
// first row, rows, first grouped position) was written by the scan.
MW4_DEV TileInfo tile_from(const GemmArgs& a, int4 bi, int m) {
    TileInfo ti;
    ti.e = checked_index(bi.x, 0, a.E + 1, a.status);
    ti.m = m;
    // the rows it names lie inside the group's grouped positions: routed [0, T*k),
    // shared [T*k, T*k + T)
    const int lo = ti.e == a.E ? a.T * a.k : 0, hi = ti.e == a.E ? a.T * a.k + a.T : a.T * a.k;
    ti.nrows = checked_index(bi.z, 1, min(kBN, hi - lo) + 1, a.status);
    ti.r0 = checked_index(bi.y, 0, hi - lo - ti.nrows + 1, a.status);
    ti.p0 = checked_index(bi.w, lo, hi - ti.nrows + 1, a.status);
    ti.sh = (ti.e == a.E);
    ti.arow = (ti.sh ? 0 : ti.e * a.rows_e) + ti.m * kBM;
    return ti;
}
MW4_DEV TileInfo block_info(const GemmArgs& a, int rb, int m) { return tile_from(a, __ldg(a.blkinfo + rb), m); }

// E4M3: the 8-bit codes are FP8 E4M3 values instead of unsigned integers.
template <bool DUAL, int BITS, bool E4M3>
__global__ void __launch_bounds__(Geo<DUAL, BITS>::kThreads, 1)
grouped_w4_gemm_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ CUtensorMap map0r,
                       const __grid_constant__ CUtensorMap map1r, const __grid_constant__ CUtensorMap map0s,
                       const __grid_constant__ CUtensorMap map1s, const __grid_constant__ CUtensorMap mapb,
                       const __grid_constant__ CUtensorMap mapbs) {
    static_assert(!E4M3 || BITS == 8, "E4M3 codes are one byte each");
    constexpr bool PRE = BITS == 16;   // fp16 weights from a separate pass: A from shared memory
    using GG = Geo<DUAL, BITS>;
    constexpr uint32_t kCodesBytes = GG::kCodesBytes;
    constexpr int kCodeWords = kGK * BITS / 32;   // code words per row per step
    constexpr int NMAT = GG::NMAT, SC = GG::SC, SB = GG::SB, SA = GG::SA;
    griddep_wait();               // programmatic dependent launch: nothing is touched before the
    griddep_launch_dependents();  // previous kernel has completed; the next one may be scheduled
    const int ntiles = checked_index(a.ntiles[0], 0, a.max_blocks * a.M + 1, a.status);
    const int G = a.K / kGroup, nK = a.K / kGK;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align1024(smem_raw);
    uint8_t* bring = base;                                   // [SB][kTileBytes], 1024-aligned stages
    uint8_t* cring = bring + (size_t)SB * kTileBytes;        // [SC][NMAT][kCodesBytes]
    auto B_of = [&](int s) { return bring + (size_t)s * kTileBytes; };
    auto C_of = [&](int s, int mat) {
        return reinterpret_cast<const uint8_t*>(cring + (size_t)s * GG::C_STAGE + mat * kCodesBytes);
    };
    float* col_scale = reinterpret_cast<float*>(cring + (size_t)SC * GG::C_STAGE);   // [2][kBN]
    uint64_t* bars = reinterpret_cast<uint64_t*>(col_scale + 2 * kBN);
    uint64_t* c_full = bars;
    uint64_t* c_empty = c_full + SC;
    uint64_t* b_full = c_empty + SC;
    uint64_t* b_empty = b_full + SB;
    uint64_t* a_full = b_empty + SB;
    uint64_t* a_empty = a_full + SA;
    uint64_t* acc_full = a_empty + SA;
    uint64_t* acc_empty = acc_full + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_empty + 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2) + 1;

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        for (int s = 0; s < SC; ++s) {
            mbar_init(&c_full[s], 1);
            mbar_init(&c_empty[s], PRE ? 1 : 32 * GG::kDeqWarps);   // PRE: freed by the MMAs' commit
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&a_full[s], 32 * GG::kDeqWarps);
            mbar_init(&a_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 32 * GG::kEpiWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == GG::kMmaWarp) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *tmem_slot;

    if (warp == GG::kProdWarp) {
        // ------------------------------------------------------------ TMA producer: codes (warp-uniform)
        // Per step: the packed codes of each matrix (128 weight rows x 16 words).
        if (lane == 0) {
            prefetch_tensormap(&map0r);
            prefetch_tensormap(&map0s);
            if (DUAL) { prefetch_tensormap(&map1r); prefetch_tensormap(&map1s); }
        }
        int gk = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const UnitInfo u = unit_info(a, t);
            const TileInfo ti = block_info(a, u.b0, u.m);
            const CUtensorMap* m0 = ti.sh ? &map0s : &map0r;
            const CUtensorMap* m1 = ti.sh ? &map1s : &map1r;
            for (int ks = 0; ks < nK; ++ks, ++gk) {
                const int s = gk % SC;
                if (!mbar_wait_warp(&c_empty[s], ((gk / SC) & 1) ^ 1, abort_flag, a.status)) { ok = false; break; }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&c_full[s], NMAT * kCodesBytes);
                    if (PRE) {   // two 64-column fp16 sub-tiles per matrix
                        for (int mat = 0; mat < NMAT; ++mat) {
                            uint8_t* dst = const_cast<uint8_t*>(C_of(s, mat));
                            tma_load_2d(dst, mat ? m1 : m0, ks * kGK, ti.arow, &c_full[s]);
                            tma_load_2d(dst + kSubBytes, mat ? m1 : m0, ks * kGK + 64, ti.arow, &c_full[s]);
                        }
                    } else {
                        tma_load_2d(const_cast<uint8_t*>(C_of(s, 0)), m0, ks * kCodeWords, ti.arow, &c_full[s]);
                        if (DUAL) tma_load_2d(const_cast<uint8_t*>(C_of(s, 1)), m1, ks * kCodeWords, ti.arow, &c_full[s]);
                    }
                }
            }
        }
    } else if (warp == GG::kProdBWarp) {
        // ------------------------------------------------------------ TMA producer: B rows (warp-uniform)
        // Per step: the step's 128 columns of the tile's B rows (two 64-column
        // sub-tiles).
        if (lane == 0) {
            prefetch_tensormap(&mapb);
            prefetch_tensormap(&mapbs);
        }
        int gk = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const UnitInfo u = unit_info(a, t);
            for (int r = 0; r < u.nb && ok; ++r) {
                const TileInfo ti = block_info(a, u.b0 + r, u.m);
                const CUtensorMap* mb = ti.sh ? &mapbs : &mapb;
                // gate/up's shared rows are rows r0.. of x16; every other B row block
                // starts at its first grouped position
                const int brow = (DUAL && ti.sh) ? ti.r0 : ti.p0;
                for (int ks = 0; ks < nK; ++ks, ++gk) {
                    const int s = gk % SB;
                    if (!mbar_wait_warp(&b_empty[s], ((gk / SB) & 1) ^ 1, abort_flag, a.status)) { ok = false; break; }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&b_full[s], kTileBytes);
                        tma_load_2d(B_of(s), mb, ks * kGK, brow, &b_full[s]);
                        tma_load_2d(B_of(s) + kSubBytes, mb, ks * kGK + 64, brow, &b_full[s]);
                    }
                }
            }
        }
    } else if (warp == GG::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer (warp-uniform, one lane issues)
        // ga counts A steps (one per K step of a unit), gb B steps (one per K step of
        // each row block of a unit)
        // The records are software-pipelined so that no tile waits on a global load:
        // the unit record two items ahead and, one lane per row block, the row-block
        // records of the next item are requested while an item runs.
        int ga = 0, gb = 0, it = 0;
        bool ok = true;
        int2 ur_c = unit_rec(a, blockIdx.x, ntiles), ur_n = unit_rec(a, blockIdx.x + gridDim.x, ntiles);
        int4 blk_c = lane < ur_c.y ? __ldg(a.blkinfo + ur_c.x + lane) : make_int4(0, 0, 0, 0);
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const int2 ur_nn = unit_rec(a, t + 2 * gridDim.x, ntiles);
            const int4 blk_n = lane < ur_n.y ? __ldg(a.blkinfo + ur_n.x + lane) : make_int4(0, 0, 0, 0);
            const int um = t % a.M, unb = ur_c.y;
            for (int r = 0; r < unb && ok; ++r, ++it) {
                int4 bi;
                bi.x = __shfl_sync(0xffffffffu, blk_c.x, r);
                bi.y = __shfl_sync(0xffffffffu, blk_c.y, r);
                bi.z = __shfl_sync(0xffffffffu, blk_c.z, r);
                bi.w = __shfl_sync(0xffffffffu, blk_c.w, r);
                const TileInfo ti = tile_from(a, bi, um);
                const int nmma = ((ti.nrows + 15) / 16) * 16;
                const uint32_t idesc = umma_idesc_f16(kBM, nmma);
                const int b = it % GG::ACC_BUFS, use = it / GG::ACC_BUFS;
                ok = mbar_wait_warp(&acc_empty[b], (use & 1) ^ 1, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t dacc = taddr + b * GG::ACC_COLS;
                for (int ks = 0; ks < nK; ++ks, ++gb) {
                    const int sb = gb % SB, ka = ga + ks, sa = ka % SA, sc = gb % SC;
                    // A from the dequantisers (a_full, waited on by the unit's first row
                    // block), or PRE from the TMA into the codes ring (c_full; one row block
                    // per unit, so A steps are B steps); B from the TMA (b_full)
                    ok = (PRE ? mbar_wait_warp(&c_full[sc], (gb / SC) & 1, abort_flag, a.status)
                              : (r > 0 || mbar_wait_warp(&a_full[sa], (ka / SA) & 1, abort_flag, a.status))) &&
                         mbar_wait_warp(&b_full[sb], (gb / SB) & 1, abort_flag, a.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t atm = taddr + GG::A_TMEM0 + sa * GG::A_COLS;
                    const uint64_t bdesc0 = umma_desc_sw128(smem_u32(B_of(sb)));
                    const uint64_t bdesc1 = umma_desc_sw128(smem_u32(B_of(sb) + kSubBytes));
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk) {
                        // K=16 slice kk: sub-tile kk/4, +32 bytes per slice within it (+2 in the address field)
                        const uint64_t bd = (kk < 4 ? bdesc0 : bdesc1) + 2 * (kk & 3);
#pragma unroll
                        for (int mat = 0; mat < NMAT; ++mat) {
                            if (PRE) {
                                const uint8_t* at = C_of(sc, mat) + (kk < 4 ? 0 : kSubBytes);
                                umma_f16_elect(dacc + mat * 128, umma_desc_sw128(smem_u32(at)) + 2 * (kk & 3), bd,
                                               idesc, (ks | kk) != 0);
                            } else {
                                umma_f16_ts_elect(dacc + mat * 128, atm + mat * (kGK / 2) + kk * 8, bd, idesc,
                                                  (ks | kk) != 0);
                            }
                        }
                    }
                    umma_commit_elect(&b_empty[sb]);   // gate/up: also frees A slot sa (see the dequantiser)
                    if (PRE) umma_commit_elect(&c_empty[sc]);
                    else if (!DUAL && r == unb - 1) umma_commit_elect(&a_empty[sa]);   // the unit's last use of A slot sa
                }
                if (ok) umma_commit_elect(&acc_full[b]);
            }
            ga += nK;
            ur_c = ur_n;
            ur_n = ur_nn;
            blk_c = blk_n;
        }
    } else if (warp < GG::kEpiWarp0) {
        // ------------------------------------------------------------ dequantisation: one weight row per thread
        if constexpr (!PRE) {   // PRE: the weights are fp16 already
            const int td = tid - 32 * GG::kDeqWarp0, row = td % 128;
            const int mat = DUAL ? td / 128 : 0, hsel = DUAL ? -1 : td / 128;   // down: which group of the step
            // swizzle phase of this row's 16-byte code chunks (64-byte rows for 4-bit
            // codes, 128-byte rows for 8-bit)
            const int sw = BITS == 8 ? (row & 7) : ((row >> 1) & 3);
            const bool chunked = (G % 8) == 0;
            int gk = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const UnitInfo u = unit_info(a, t);
                const TileInfo ti = block_info(a, u.b0, u.m);   // the unit's group and weight rows
                const uint16_t* sp = (mat == 0 ? (ti.sh ? a.s0s : a.s0r) : (ti.sh ? a.s1s : a.s1r)) + (size_t)(ti.arow + row) * G;
                const uint16_t* bp = (mat == 0 ? (ti.sh ? a.b0s : a.b0r) : (ti.sh ? a.b1s : a.b1r)) + (size_t)(ti.arow + row) * G;
                uint4 sq = make_uint4(0, 0, 0, 0), bq = sq, sqn = sq, bqn = sq;
                if (chunked) {
                    sq = __ldg(reinterpret_cast<const uint4*>(sp));
                    bq = __ldg(reinterpret_cast<const uint4*>(bp));
                }
                for (int k4 = 0; k4 < nK; k4 += 4) {   // four steps = eight groups per scale/bias load
                    if (chunked && k4 + 4 < nK) {
                        sqn = __ldg(reinterpret_cast<const uint4*>(sp + 2 * (k4 + 4)));
                        bqn = __ldg(reinterpret_cast<const uint4*>(bp + 2 * (k4 + 4)));
                    }
    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int ks = k4 + j;
                        if (ks >= nK) break;
                        uint32_t s2w, b2w;   // the step's two groups, bf16 pairs (low half first)
                        if (chunked) {
                            s2w = (j == 0 ? sq.x : j == 1 ? sq.y : j == 2 ? sq.z : sq.w);
                            b2w = (j == 0 ? bq.x : j == 1 ? bq.y : j == 2 ? bq.z : bq.w);
                        } else {
                            s2w = (uint32_t)sp[2 * ks] | ((uint32_t)sp[2 * ks + 1] << 16);
                            b2w = (uint32_t)bp[2 * ks] | ((uint32_t)bp[2 * ks + 1] << 16);
                        }
                        const int sc = gk % SC, sa = gk % SA;
                        // A slot sa last served A step gk - SA.  Down: a_empty fires once the
                        // MMAs of every row block of that step's unit are done.  Gate/up (one row
                        // block per unit, A step = B step): the commit on b_empty of that step
                        // does (SA <= SB, so that barrier cannot have moved on by a further
                        // phase meanwhile), and no separate commit is spent.
                        if constexpr (DUAL) {
                            // gate/up: the codes and the A slot first, then the step's code chunks
                            // requested together (a tensor-memory store orders later shared-memory
                            // loads behind it), then each quad rebuilt and stored in turn (measured
                            // faster than rebuilding any part of the step before the slot wait)
                            ok = mbar_wait(&c_full[sc], (gk / SC) & 1, abort_flag, a.status) &&
                                 (gk < SA || mbar_wait(&b_empty[(gk - SA) % SB], ((gk - SA) / SB) & 1, abort_flag,
                                                       a.status));
                            if (!ok) break;
                            const uint8_t* cr = C_of(sc, mat) + row * GG::kCodesRowBytes;
                            constexpr int kCPQ = BITS == 8 ? 2 : 1;   // 16-byte chunks per 32 columns
                            uint4 wc[2][2][kCPQ];
#pragma unroll
                            for (int grp = 0; grp < 2; ++grp) {
#pragma unroll
                                for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                                    for (int hh2 = 0; hh2 < kCPQ; ++hh2) {
                                        const int c = kCPQ * (2 * grp + qq) + hh2;
                                        wc[grp][qq][hh2] = *reinterpret_cast<const uint4*>(cr + ((c ^ sw) << 4));
                                    }
                            }
                            tc_fence_after();   // the MMAs that read this A slot have completed
                            // this thread's weight row -> its TMEM lane, 64 columns of fp16 pairs, in quads of 16
                            const uint32_t tdst =
                                taddr + ((uint32_t)(row & ~31) << 16) + GG::A_TMEM0 + sa * GG::A_COLS + mat * (kGK / 2);
    #pragma unroll
                            for (int grp = 0; grp < 2; ++grp) {
                                const float sf = bf16_bits_to_float((uint16_t)(grp ? (s2w >> 16) : (s2w & 0xFFFFu)));
                                const float bf = bf16_bits_to_float((uint16_t)(grp ? (b2w >> 16) : (b2w & 0xFFFFu)));
                                // the group's rebuilt weights |s q + b| must stay within fp16 (q <= the
                                // largest code magnitude: 15, 255, or 448 for E4M3)
                                constexpr float kQmax = BITS == 4 ? 15.f : (E4M3 ? 448.f : 255.f);
                                if (!(fmaf(fabsf(sf), kQmax, fabsf(bf)) <= 65504.f)) raise_status(a.status, MOE_W4_STATUS_FP16_RANGE);
                                const __half s_h = __float2half_rn(sf), s_h16 = __float2half_rn(sf * 0.0625f);
                                const __half b_h = __float2half_rn(bf);
                                const __half2 s2 = __halves2half2(s_h, s_h), s2_16 = __halves2half2(s_h16, s_h16);
                                const __half2 b2 = __halves2half2(b_h, b_h);
    #pragma unroll
                                for (int qq = 0; qq < 2; ++qq) {   // 32 columns of the group -> 16 TMEM columns
                                    const int q = 2 * grp + qq;
                                    uint32_t o[16];
                                    if (BITS == 8) {   // two 16-byte chunks of four words
    #pragma unroll
                                        for (int hh2 = 0; hh2 < 2; ++hh2) {
                                            const uint4 w = wc[grp][qq][hh2 % kCPQ];
                                            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    #pragma unroll
                                            for (int wi = 0; wi < 4; ++wi) {
                                                uint32_t q2[2];
                                                if (E4M3)
                                                    dequant_e4m3x4_f16(words[wi], s2, b2, q2);
                                                else
                                                    dequant4x8_f16(words[wi], s2, b2, q2);
                                                o[8 * hh2 + 2 * wi] = q2[0];
                                                o[8 * hh2 + 2 * wi + 1] = q2[1];
                                            }
                                        }
                                    } else {           // one 16-byte chunk of four words
                                        const uint4 w = wc[grp][qq][0];
                                        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    #pragma unroll
                                        for (int wi = 0; wi < 4; ++wi) {
                                            uint32_t q4[4];
                                            dequant8_f16(words[wi], s2, s2_16, b2, q4);
                                            o[4 * wi] = q4[0]; o[4 * wi + 1] = q4[1]; o[4 * wi + 2] = q4[2]; o[4 * wi + 3] = q4[3];
                                        }
                                    }
                                    tmem_st16(tdst + 16 * q, o);
                                }
                            }
                        } else {
                            // down: the step rebuilt in registers first, while the MMAs of the
                            // previous unit may still read A slot sa, then stored once it is free
                            if (!(ok = mbar_wait(&c_full[sc], (gk / SC) & 1, abort_flag, a.status))) break;
                            const uint8_t* cr = C_of(sc, mat) + row * GG::kCodesRowBytes;
                            constexpr int kCPQ = BITS == 8 ? 2 : 1;   // 16-byte chunks per 32 columns
                            uint4 wc[2][kCPQ];
#pragma unroll
                            for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                                for (int hh2 = 0; hh2 < kCPQ; ++hh2) {
                                    const int c = kCPQ * (2 * hsel + qq) + hh2;
                                    wc[qq][hh2] = *reinterpret_cast<const uint4*>(cr + ((c ^ sw) << 4));
                                }
                            const float sf = bf16_bits_to_float((uint16_t)(hsel ? (s2w >> 16) : (s2w & 0xFFFFu)));
                            const float bf = bf16_bits_to_float((uint16_t)(hsel ? (b2w >> 16) : (b2w & 0xFFFFu)));
                            constexpr float kQmax = BITS == 4 ? 15.f : (E4M3 ? 448.f : 255.f);
                            if (!(fmaf(fabsf(sf), kQmax, fabsf(bf)) <= 65504.f)) raise_status(a.status, MOE_W4_STATUS_FP16_RANGE);
                            const __half s_h = __float2half_rn(sf), s_h16 = __float2half_rn(sf * 0.0625f);
                            const __half b_h = __float2half_rn(bf);
                            const __half2 s2 = __halves2half2(s_h, s_h), s2_16 = __halves2half2(s_h16, s_h16);
                            const __half2 b2 = __halves2half2(b_h, b_h);
                            uint32_t o[2][16];
#pragma unroll
                            for (int qq = 0; qq < 2; ++qq) {
                                if (BITS == 8) {
#pragma unroll
                                    for (int hh2 = 0; hh2 < 2; ++hh2) {
                                        const uint4 w = wc[qq][hh2 % kCPQ];
                                        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                        for (int wi = 0; wi < 4; ++wi) {
                                            uint32_t q2[2];
                                            if (E4M3)
                                                dequant_e4m3x4_f16(words[wi], s2, b2, q2);
                                            else
                                                dequant4x8_f16(words[wi], s2, b2, q2);
                                            o[qq][8 * hh2 + 2 * wi] = q2[0];
                                            o[qq][8 * hh2 + 2 * wi + 1] = q2[1];
                                        }
                                    }
                                } else {
                                    const uint4 w = wc[qq][0];
                                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                    for (int wi = 0; wi < 4; ++wi) {
                                        uint32_t q4[4];
                                        dequant8_f16(words[wi], s2, s2_16, b2, q4);
                                        o[qq][4 * wi] = q4[0]; o[qq][4 * wi + 1] = q4[1];
                                        o[qq][4 * wi + 2] = q4[2]; o[qq][4 * wi + 3] = q4[3];
                                    }
                                }
                            }
                            if (!(ok = mbar_wait(&a_empty[sa], ((gk / SA) & 1) ^ 1, abort_flag, a.status))) break;
                            tc_fence_after();   // the MMAs that read this A slot have completed
                            const uint32_t tdst =
                                taddr + ((uint32_t)(row & ~31) << 16) + GG::A_TMEM0 + sa * GG::A_COLS;
#pragma unroll
                            for (int qq = 0; qq < 2; ++qq) tmem_st16(tdst + 16 * (2 * hsel + qq), o[qq]);
                        }
                        tmem_wait_st();
                        mbar_arrive(&c_empty[sc]);   // this thread's codes of the step are read
                        tc_fence_before();
                        mbar_arrive(&a_full[sa]);
                        ++gk;
                    }
                    if (!ok) break;
                    sq = sqn;
                    bq = bqn;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue: TMEM -> registers -> global
        const int ew = warp - GG::kEpiWarp0, q = ew & 3, half = ew >> 2;
        const int et = tid - 32 * GG::kEpiWarp0;
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const UnitInfo un = unit_info(a, t);
            for (int r = 0; r < un.nb; ++r, ++it) {
                const TileInfo ti = block_info(a, un.b0 + r, un.m);
                const int b = it % GG::ACC_BUFS, use = it / GG::ACC_BUFS, cb = it & 1;
                // gate/up: the weight of each column of the tile (its routing weight, or the
                // shared gate) is applied to h, so that the down projection's output needs
                // none; fetched while the MMAs run (two buffers: a thread writes a buffer
                // only after every thread has passed the previous tile's barrier)
                if (DUAL) {
                    if (et < ti.nrows)
                        col_scale[cb * kBN + et] =
                            ti.sh ? a.gamma[ti.r0 + et]
                                  : a.topk_w[checked_index(a.perm[ti.p0 + et], 0, a.T * a.k, a.status)];
                    asm volatile("bar.sync 2, 256;" ::: "memory");
                }
                ok = mbar_wait(&acc_full[b], use & 1, abort_flag, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t lane_addr = taddr + b * GG::ACC_COLS + ((uint32_t)(q * 32) << 16);
                // h is the K operand of the down projection: store it in chunk order
                const int orow = ti.m * kBM + q * 32 + lane;
                const bool ko8 = PRE ? a.k_order8 != 0 : BITS == 8;   // the layer's codes, not the fp16 copy
                const int ocol = DUAL ? ((orow & ~7) | (ko8 ? chunk8_pos_of_col(orow & 7) : chunk_pos_of_col(orow & 7)))
                                      : orow;
                for (int c0 = half * 16; c0 < ti.nrows; c0 += 32) {
                    uint32_t g[16], u[16];
                    tmem_ld16(lane_addr + c0, g);
                    if (DUAL) tmem_ld16(lane_addr + 128 + c0, u);
                    tmem_wait_ld();
                    // column n of the tile is grouped row p0 + n: one pointer per chunk, rows
                    // out_cols apart; a full chunk runs without per-element branches
                    uint16_t* op = a.out + (size_t)(ti.p0 + c0) * a.out_cols + ocol;
                    float cs[16];
                    if (DUAL) {
                        const float4* c4 = reinterpret_cast<const float4*>(col_scale + cb * kBN + c0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 f = c4[i];
                            cs[4 * i] = f.x; cs[4 * i + 1] = f.y; cs[4 * i + 2] = f.z; cs[4 * i + 3] = f.w;
                        }
                    }
                    // range check on the running maximum of |v| (the values are finite: fp16
                    // operands, fp32 sums far below the fp32 limit)
                    float vmax = 0.f;
                    auto emit = [&](int j) {
                        const float v = DUAL ? silu_tanh(__uint_as_float(g[j])) * __uint_as_float(u[j]) * cs[j]
                                             : __uint_as_float(g[j]);
                        vmax = fmaxf(vmax, fabsf(v));
                        op[(size_t)j * a.out_cols] = __half_as_ushort(__float2half_rn(v));
                    };
                    if (c0 + 16 <= ti.nrows) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) emit(j);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (j < ti.nrows - c0) emit(j);
                    }
                    if (!(vmax <= 65504.f)) raise_status(a.status, MOE_W4_STATUS_FP16_RANGE);
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[b]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == GG::kMmaWarp) tmem_dealloc(taddr, 512);
}

// xg[p] = x16[perm[p] / k] for the T*k routed grouped positions p: one warp per
// row, 16-byte loads and stores, eight in flight per lane.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x16,
                                                          const int32_t* __restrict__ perm,
                                                          uint16_t* __restrict__ xg, int nrows, int H, int k,
                                                          unsigned int* status) {
    const int p = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
    griddep_wait();               // programmatic dependent launch: nothing is touched before the
    griddep_launch_dependents();  // previous kernel has completed; the next one may be scheduled
    if (p >= nrows) return;
    const int t = checked_index(__ldg(perm + p), 0, nrows, status) / k;
    const uint4* src = reinterpret_cast<const uint4*>(x16 + (size_t)t * H);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)p * H);
    const int n = H / 8;
    for (int c0 = lane; c0 < n; c0 += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c0 + 32 * u < n) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c0 + 32 * u < n) dst[c0 + 32 * u] = v[u];
    }
}

// out[t] = bf16( sum_j ys[inv[t*k + j]] + ys[T*k + t] ) with ys in fp16 and
// the sum in fp32, slots in order then the shared row; 8 columns per thread.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ ys,
                                                      const int32_t* __restrict__ inv, uint16_t* __restrict__ out,
                                                      int T, int H, int k, unsigned int* status) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int per_row = H / 8;
    griddep_wait();               // programmatic dependent launch: nothing is touched before the
    griddep_launch_dependents();  // previous kernel has completed; the next one may be scheduled
    if (i >= (size_t)T * per_row) return;
    const int t = (int)(i / per_row), c = (int)(i % per_row) * 8;
    // all k + 1 rows requested before the first is added (k <= 8), then added in order
    uint4 v[9];
#pragma unroll
    for (int j = 0; j < 9; ++j) {
        if (j > k) break;
        const size_t p = (j < k) ? (size_t)checked_index(inv[(size_t)t * k + j], 0, T * k, status) : (size_t)T * k + t;
        v[j] = __ldg(reinterpret_cast<const uint4*>(ys + p * H + c));
    }
    float acc[8] = {};
#pragma unroll
    for (int j = 0; j < 9; ++j) {
        if (j > k) break;
        const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
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

// One grouped GEMM launch (the shared-memory size is raised once per device
// and instance).
template <bool DUAL, int BITS, bool E4M3>
static cudaError_t launch_gemm(const GemmArgs& g, int grid, const CUtensorMap& m0r, const CUtensorMap& m1r,
                               const CUtensorMap& m0s, const CUtensorMap& m1s, const CUtensorMap& mb,
                               const CUtensorMap& mbs, cudaStream_t st, bool pdl) {
    using GG = Geo<DUAL, BITS>;
    static bool set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!set[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(grouped_w4_gemm_kernel<DUAL, BITS, E4M3>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GG::bytes());
        if (e != cudaSuccess) return e;
        set[dev] = true;
    }
    return launch_pdl(pdl, grouped_w4_gemm_kernel<DUAL, BITS, E4M3>, dim3(grid), dim3(GG::kThreads), GG::bytes(), st, g, m0r,
                      m1r, m0s, m1s, mb, mbs);
}

cudaError_t launch_grouped_ffn(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out, const PrefillWs& p,
                               cudaStream_t st, const uint16_t* const* w16) {
    const int bits = code_bits_of(L);
    const bool e4m3 = codes_e4m3(L);   // validated: only with 8-bit codes
    const int H = L.H, I = L.I, E = L.E, k = L.top_k;
    const uint64_t rows_all = (uint64_t)T * k + T;
    CUtensorMap mg, mu, msg, msu, md, msd, mh, mxg, mx;
    const auto U32 = CU_TENSOR_MAP_DATA_TYPE_UINT32;
    // code rows of one step: 64 bytes (4-bit codes) or 128 bytes (8-bit), swizzled
    // to match so that the per-row reads are bank-conflict free
    const auto SWC = bits == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const uint32_t cw = kGK * bits / 32;            // code words per row per step
    const int wH = H * bits / 32, wI = I * bits / 32;   // code words per row of gate/up and of down
    bool ok = make_map(&mg, U32, 4, L.gate.codes, (uint64_t)E * I, wH, kBM, cw, SWC) &&
              make_map(&mu, U32, 4, L.up.codes, (uint64_t)E * I, wH, kBM, cw, SWC) &&
              make_map(&msg, U32, 4, L.sh_gate.codes, I, wH, kBM, cw, SWC) &&
              make_map(&msu, U32, 4, L.sh_up.codes, I, wH, kBM, cw, SWC) &&
              make_map(&md, U32, 4, L.down.codes, (uint64_t)E * H, wI, kBM, cw, SWC) &&
              make_map(&msd, U32, 4, L.sh_down.codes, H, wI, kBM, cw, SWC) &&
              make_map(&mh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.hh, rows_all, I, kBN, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&mxg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.xg, (uint64_t)T * k, H, kBN, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.x16, (uint64_t)T, H, kBN, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (w16) {   // fp16 weights from the separate pass: 64-column boxes, as the B tiles
        const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
        ok = ok && make_map(&mg, F16, 2, w16[0], (uint64_t)E * I, H, kBM, 64, SW) &&
             make_map(&mu, F16, 2, w16[1], (uint64_t)E * I, H, kBM, 64, SW) &&
             make_map(&md, F16, 2, w16[2], (uint64_t)E * H, I, kBM, 64, SW) &&
             make_map(&msg, F16, 2, w16[3], I, H, kBM, 64, SW) && make_map(&msu, F16, 2, w16[4], I, H, kBM, 64, SW) &&
             make_map(&msd, F16, 2, w16[5], H, I, kBM, 64, SW);
    }
    if (!ok) return cudaErrorInvalidValue;

    int nsm = 0;
    {
        int dv = 0;
        cudaGetDevice(&dv);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dv);
        if (nsm <= 0) nsm = 148;
    }

    GemmArgs a{};
    a.ntiles = p.ntiles; a.offsets = p.offsets; a.perm = p.perm;
    a.topk_w = p.topk_w; a.gamma = p.gamma;
    a.E = E; a.k = k; a.T = T; a.H = H; a.status = p.status; a.k_order8 = bits == 8;
    a.max_blocks = p.max_tiles_gu / (I / kBM);

    // gate/up: A = Wg, Wu rows (I per expert), K = H, out = hh [.][I]
    a.blkinfo = p.blkinfo; a.unitinfo = nullptr; a.M = I / kBM;
    a.s0r = L.gate.scales; a.b0r = L.gate.biases; a.s1r = L.up.scales; a.b1r = L.up.biases;
    a.s0s = L.sh_gate.scales; a.b0s = L.sh_gate.biases; a.s1s = L.sh_up.scales; a.b1s = L.sh_up.biases;
    a.out = p.hh; a.K = H; a.rows_e = I; a.out_cols = I;
    // persistent: one CTA per SM (never more CTAs than the largest tile count)
    const int grid_gu = p.max_tiles_gu < nsm ? p.max_tiles_gu : nsm;
    const int nrg = T * k;
    cudaError_t e = launch_pdl(pdl_for(T), gather_rows_kernel, dim3((unsigned)((nrg + 7) / 8)), dim3(256), 0, st, p.x16, p.perm,
                               p.xg, nrg, H, k, p.status);
    if (e != cudaSuccess) return e;
    trace_mark(st, 4);
    e = w16   ? launch_gemm<true, 16, false>(a, grid_gu, mg, mu, msg, msu, mxg, mx, st, pdl_for(T))
                  : e4m3  ? launch_gemm<true, 8, true>(a, grid_gu, mg, mu, msg, msu, mxg, mx, st, pdl_for(T))
                  : bits == 8 ? launch_gemm<true, 8, false>(a, grid_gu, mg, mu, msg, msu, mxg, mx, st, pdl_for(T))
                              : launch_gemm<true, 4, false>(a, grid_gu, mg, mu, msg, msu, mxg, mx, st, pdl_for(T));
    if (e != cudaSuccess) return e;
    trace_mark(st, 5);

    // down: A = Wd rows (H per expert), K = I, B = hh rows, out = ys [.][H]
    GemmArgs b = a;
    b.M = H / kBM; b.ntiles = p.ntiles + 1; b.unitinfo = p.unitinfo;   // fp16 weights: one-block units (du = 1)
    b.s0r = L.down.scales; b.b0r = L.down.biases; b.s1r = nullptr; b.b1r = nullptr;
    b.s0s = L.sh_down.scales; b.b0s = L.sh_down.biases; b.s1s = nullptr; b.b1s = nullptr;
    b.out = p.ys; b.K = I; b.rows_e = H; b.out_cols = H;
    const int grid_dn = p.max_tiles_dn < nsm ? p.max_tiles_dn : nsm;
    e = w16   ? launch_gemm<false, 16, false>(b, grid_dn, md, md, msd, msd, mh, mh, st, pdl_for(T))
      : e4m3  ? launch_gemm<false, 8, true>(b, grid_dn, md, md, msd, msd, mh, mh, st, pdl_for(T))
      : bits == 8 ? launch_gemm<false, 8, false>(b, grid_dn, md, md, msd, msd, mh, mh, st, pdl_for(T))
                  : launch_gemm<false, 4, false>(b, grid_dn, md, md, msd, msd, mh, mh, st, pdl_for(T));
    if (e != cudaSuccess) return e;
    trace_mark(st, 6);

    const size_t nthr = (size_t)T * (H / 8);
    e = launch_pdl(pdl_for(T), combine_kernel, dim3((unsigned)((nthr + 255) / 256)), dim3(256), 0, st, p.ys, p.inv, out, T, H, k,
                   p.status);
    if (e != cudaSuccess) return e;
    trace_mark(st, 7);
    return cudaGetLastError();
}

}  // namespace mw4
