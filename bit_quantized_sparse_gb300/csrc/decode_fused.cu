// Fused batch-1 decode: the whole layer for one token in one launch.
// ("Optimizing on-device inference for Apple Silicon", sections "Optimise the
// single-row weight path" -- groups of threads cooperate on outputs while
// reading different parts of the weight matrix -- and "Reduce intermediate
// state and traffic" -- gate/up projections fused with the gated activation,
// the output projection fused with the routing scores and the shared expert.)
//
// Grid: (k+1) clusters of kCS CTAs.  Cluster j < k serves the j-th selected
// expert, cluster k the shared expert.  CTA r of a cluster owns gate/up rows
// [r*I/kCS, (r+1)*I/kCS) and down rows [r*H/kCS, (r+1)*H/kCS) of its expert.
//
//   1. router: every CTA sums x . W_r over its own 1/((k+1) kCS) slice of the
//      H rows for all E experts; the slices are reduced in each cluster
//      through distributed shared memory, and the k+1 cluster sums are
//      exchanged through global memory (bounded wait: all clusters are
//      co-resident, one CTA per SM).  Each CTA then selects the top-k.
//      The shared cluster does not wait for the routing: it starts loading its
//      weights as soon as its own router reads are done.
//   2. TMA loads the CTA's slices of the packed codes (128-byte swizzle) and
//      its scales/biases; the gate/up slices are consumed box by box as they
//      land.
//   3. gate/up GEMV on the tensor cores as a dot-product engine: mma.sync
//      m16n8k16 with A = bf16(128 + q) built from the codes by one bitwise op
//      per pair, B = x (exact in bf16), fp32 accumulation per 64-column group;
//      then w = s*(acc - 128*sum(x)) + b*sum(x).  SwiGLU in fp32.
//   4. h is exchanged inside the cluster (distributed shared memory).
//   5. down GEMV the same way with fp16 (1024 + q) x fp16 h, scaled by the
//      routing weight (or the shared gate), written per expert.
//   6. per block of output rows, the last of the k+1 CTAs to finish adds the
//      k+1 expert outputs in slot order and writes bf16 out.
// No step waits on another CTA except the bounded router exchange and the
// hardware cluster barriers.
#include "common.cuh"
#include "internal.h"

namespace mw4 {

constexpr int kCS = 8;          // CTAs per cluster
constexpr int kFThreads = 512;  // 16 warps
constexpr int kFWarps = kFThreads / 32;
constexpr int kMaxSlots = 9;   // k + 1 <= 9

struct FusedArgs {
    const uint16_t* x;          // [H] bf16
    const float* router_w;      // [H][E]
    const float* router_bias;   // [E] or NULL
    const float* shared_gate;   // [H]
    const uint16_t* gs; const uint16_t* gb; const uint16_t* us; const uint16_t* ub;   // routed gate/up s, b
    const uint16_t* ds; const uint16_t* db;                                             // routed down s, b
    const uint16_t* sgs; const uint16_t* sgb; const uint16_t* sus; const uint16_t* sub; // shared
    const uint16_t* sds; const uint16_t* sdb;
    float* cpart;               // [k+1][E] cluster partial scores
    float* ybuf;                // [k+1][H] weighted expert outputs
    int32_t* idx_out;           // [k] (for inspection)
    float* w_out;               // [k]
    float* gamma_out;           // [1]
    uint16_t* out;              // [H] bf16
    Ctrl* ctrl;
    int H, E, I, k;
};

// smem carve-up (byte offsets from a 1024-aligned base), computed on both sides
struct FusedSmem {
    uint32_t gcodes, ucodes, dcodes, gsb, usb, dsb, xperm, xsum, part, logits, gsum, usum, hloc, hperm, hsum,
        red, misc, total;
    int RG, RD;
    __host__ __device__ FusedSmem(int H, int E, int I) {
        RG = I / kCS;
        RD = H / kCS;
        uint32_t o = 0;
        auto take = [&](uint32_t bytes, uint32_t align) {
            o = (o + align - 1) / align * align;
            const uint32_t at = o;
            o += bytes;
            return at;
        };
        gcodes = take(RG * H / 2, 1024);
        ucodes = take(RG * H / 2, 1024);
        dcodes = take(RD * I / 2, 1024);
        gsb = take(2 * RG * (H / 64) * 2, 16);   // scales then biases
        usb = take(2 * RG * (H / 64) * 2, 16);
        dsb = take(2 * RD * (I / 64) * 2, 16);
        xperm = take(H * 2, 16);
        xsum = take(H / 64 * 4, 16);
        part = take(E * 4, 16);
        logits = take(E * 4, 16);
        gsum = take(RG * 4, 16);
        usum = take(RG * 4, 16);
        hloc = take(RG * 4, 16);
        hperm = take(I * 2, 16);
        hsum = take(I / 64 * 4, 16);
        red = part;   // K-split partials reuse the score buffers (part, logits: 2E floats) after routing
        misc = take(256, 16);
        total = o;
    }
};

// --------------------------------------------------------------------------- cluster helpers
MW4_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
MW4_DEV uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
MW4_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
MW4_DEV float ld_dsmem_f32(const void* local_ptr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_ptr)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}
MW4_DEV uint32_t ld_acquire_u32(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// --------------------------------------------------------------------------- legacy-MMA dot engine
MW4_DEV void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
MW4_DEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Codes word `wi` (0-based along the row) of row `row` inside a 128-byte
// swizzled TMA tile set: boxes of 32 words x `rows` rows, box b at b*rows*128.
MW4_DEV uint32_t sw_word(const uint8_t* base, int rows, int row, int wi) {
    const int box = wi >> 5, u = (wi >> 2) & 7, w = wi & 3;
    return *reinterpret_cast<const uint32_t*>(base + (size_t)box * rows * 128 + row * 128 + ((u ^ (row & 7)) << 4) +
                                              w * 4);
}

// One warp: rows [r0, r0+16) of a swizzled codes tile set, 64-column groups
// [grp0, grp1); B fragments from `bperm` (16 bytes per (32-column block,
// lane%4)), column sums `gsum` (per 64 columns), scale/bias tables
// [rows][ngrp_row].  Adds the dot products of rows r0+g and r0+g+8 (g =
// lane/4) to acc0/acc1.  Two groups are in flight at a time so that the
// chained MMAs of one group overlap the other's.
MW4_DEV void w4_group_mma(const uint8_t* codes, int rows, int r0, int grp, const uint4* bperm, uint32_t magic,
                          bool f16, float (&d)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    // both rows of the thread (r0+g, r0+g+8) share the swizzle phase g; a group
    // (2 blocks of 32 columns) lies inside one box of 8 blocks
    const int blk0 = grp * 2;
    const uint8_t* row0 = codes + (size_t)(blk0 >> 3) * rows * 128 + (r0 + g) * 128 + c * 4;
    const uint8_t* row1 = row0 + 8 * 128;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int blk = blk0 + h;
        const int off = ((blk & 7) ^ g) << 4;
        const uint32_t wg = *reinterpret_cast<const uint32_t*>(row0 + off);
        const uint32_t wh = *reinterpret_cast<const uint32_t*>(row1 + off);
        const uint4 bv = bperm[blk * 4 + c];
        uint32_t a[4];
        a[0] = (wg & 0x000F000Fu) | magic;
        a[1] = (wh & 0x000F000Fu) | magic;
        a[2] = ((wg >> 4) & 0x000F000Fu) | magic;
        a[3] = ((wh >> 4) & 0x000F000Fu) | magic;
        if (f16) mma_f16_16816(d, a, bv.x, bv.y); else mma_bf16_16816(d, a, bv.x, bv.y);
        a[0] = ((wg >> 8) & 0x000F000Fu) | magic;
        a[1] = ((wh >> 8) & 0x000F000Fu) | magic;
        a[2] = ((wg >> 12) & 0x000F000Fu) | magic;
        a[3] = ((wh >> 12) & 0x000F000Fu) | magic;
        if (f16) mma_f16_16816(d, a, bv.z, bv.w); else mma_bf16_16816(d, a, bv.z, bv.w);
    }
}

template <bool F16>
MW4_DEV bool w4_gemv16(const uint8_t* codes, int rows, int r0, int grp0, int grp1, const uint4* bperm,
                       const float* gsum, const uint16_t* sc, const uint16_t* bi, int ngrp_row, float& acc0,
                       float& acc1, uint64_t* box_bars, volatile int* abort_flag, unsigned int* status) {
    const int lane = threadIdx.x & 31, g = lane >> 2;
    const uint32_t magic = F16 ? 0x64006400u : 0x43004300u;
    const float offs = F16 ? 1024.f : 128.f;
    constexpr int kIn = 4;   // groups in flight: independent MMA chains
    for (int grp = grp0; grp < grp1; grp += kIn) {
        if (box_bars) {   // 4 groups (256 columns) per TMA box
            for (int q = 0; q < kIn; ++q)
                if (grp + q < grp1 && ((grp + q) & 3) == 0 || (q == 0 && grp + q < grp1))
                    if (!mbar_wait(&box_bars[(grp + q) >> 2], 0, abort_flag, status)) return false;
        }
        float d[kIn][4];
#pragma unroll
        for (int q = 0; q < kIn; ++q) {
            d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.f;
            if (grp + q < grp1) w4_group_mma(codes, rows, r0, grp + q, bperm, magic, F16, d[q]);
        }
        // every lane of a row group holds the same column sums (B is the same for all n)
#pragma unroll
        for (int q = 0; q < kIn; ++q) {
            const int gg = grp + q;
            if (gg >= grp1) break;
            const float xs = gsum[gg];
            const float s0 = bf16_bits_to_float(sc[(r0 + g) * ngrp_row + gg]);
            const float b0 = bf16_bits_to_float(bi[(r0 + g) * ngrp_row + gg]);
            const float s1 = bf16_bits_to_float(sc[(r0 + g + 8) * ngrp_row + gg]);
            const float b1 = bf16_bits_to_float(bi[(r0 + g + 8) * ngrp_row + gg]);
            acc0 = fmaf(s0, d[q][0] - offs * xs, fmaf(b0, xs, acc0));
            acc1 = fmaf(s1, d[q][2] - offs * xs, fmaf(b1, xs, acc1));
        }
    }
    return true;
}

__global__ void __launch_bounds__(kFThreads, 1)
decode_fused_kernel(const __grid_constant__ FusedArgs a, const __grid_constant__ CUtensorMap mg,
                    const __grid_constant__ CUtensorMap mu, const __grid_constant__ CUtensorMap md,
                    const __grid_constant__ CUtensorMap msg, const __grid_constant__ CUtensorMap msu,
                    const __grid_constant__ CUtensorMap msd) {
    const int H = a.H, E = a.E, I = a.I, k = a.k;
    const FusedSmem L(H, E, I);
    const int RG = L.RG, RD = L.RD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* gcodes = sm + L.gcodes;
    uint8_t* ucodes = sm + L.ucodes;
    uint8_t* dcodes = sm + L.dcodes;
    uint16_t* gsb = reinterpret_cast<uint16_t*>(sm + L.gsb);
    uint16_t* usb = reinterpret_cast<uint16_t*>(sm + L.usb);
    uint16_t* dsb = reinterpret_cast<uint16_t*>(sm + L.dsb);
    uint32_t* xperm = reinterpret_cast<uint32_t*>(sm + L.xperm);
    float* xsum = reinterpret_cast<float*>(sm + L.xsum);
    float* part = reinterpret_cast<float*>(sm + L.part);
    float* logits = reinterpret_cast<float*>(sm + L.logits);
    float* gsum = reinterpret_cast<float*>(sm + L.gsum);
    float* usum = reinterpret_cast<float*>(sm + L.usum);
    float* hloc = reinterpret_cast<float*>(sm + L.hloc);
    uint32_t* hperm = reinterpret_cast<uint32_t*>(sm + L.hperm);
    float* hsum = reinterpret_cast<float*>(sm + L.hsum);
    float* red = reinterpret_cast<float*>(sm + L.red);
    uint8_t* misc = sm + L.misc;
    const int nbox_gu = H / 256, nbox_dn = I / 256 > 0 ? I / 256 : 1;
    uint64_t* bar_gu = reinterpret_cast<uint64_t*>(misc);               // [nbox_gu] (<= 16)
    uint64_t* bar_dn = bar_gu + 16;                                      // [1]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_dn + 1);
    int* sel_e = reinterpret_cast<int*>(bar_dn + 2);                     // selected expert of this cluster
    float* sel_w = reinterpret_cast<float*>(sel_e + 1);                  // its weight (or gamma)
    int* last_flag = reinterpret_cast<int*>(sel_e + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = (int)cluster_rank(), slot = (int)cluster_id();
    const int NC = k + 1, NG = NC * kCS, G = slot * kCS + rank;
    const bool shared_cluster = (slot == k);
    unsigned int* status = &a.ctrl->status;

    // the router's loads go out first: thread (e, half) sums half of this CTA's
    // slice of the H rows for expert e; its W_r column slice and the matching x
    // values (the same for the whole warp) land while x is prepared below
    const int rh0 = (int)((long)G * H / NG), rh1 = (int)((long)(G + 1) * H / NG);
    const int rnh = rh1 - rh0, rhalf = rnh / 2;
    const int r_e = tid % E, r_hb = (tid / E) ? rhalf : 0, r_he = (tid / E) ? rnh : rhalf;
    float rw[32], rx[32];
    if (tid < 2 * E) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const bool in = r_hb + j < r_he;
            rw[j] = in ? __ldg(a.router_w + (size_t)(rh0 + r_hb + j) * E + r_e) : 0.f;
            rx[j] = in ? bf16_bits_to_float(__ldg(a.x + rh0 + r_hb + j)) : 0.f;
        }
    }
    if (tid == 32) {   // the descriptors are fetched once, early, off the critical path
        prefetch_tensormap(&mg); prefetch_tensormap(&mu); prefetch_tensormap(&md);
        prefetch_tensormap(&msg); prefetch_tensormap(&msu); prefetch_tensormap(&msd);
    }
    if (tid == 0) {
        for (int b = 0; b < nbox_gu; ++b) mbar_init(&bar_gu[b], 1);
        mbar_init(bar_dn, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // x as permuted bf16 pairs for the B fragments, and per-64-column sums
    // (block of 32 columns, lane%4 = c): {x[8c], x[8c+4]}, {x[8c+1], x[8c+5]},
    // {x[8c+2], x[8c+6]}, {x[8c+3], x[8c+7]}
    for (int i = tid; i < H / 8; i += kFThreads) {
        const uint4 v = *reinterpret_cast<const uint4*>(a.x + i * 8);
        const uint32_t e[4] = {v.x, v.y, v.z, v.w};   // pairs (0,1) (2,3) (4,5) (6,7)
        const uint32_t q0 = __byte_perm(e[0], e[2], 0x5410), q1 = __byte_perm(e[0], e[2], 0x7632);
        const uint32_t q2 = __byte_perm(e[1], e[3], 0x5410), q3 = __byte_perm(e[1], e[3], 0x7632);
        uint4* dst = reinterpret_cast<uint4*>(xperm) + i;   // i = blk*4 + c
        *dst = make_uint4(q0, q1, q2, q3);
    }
    __syncthreads();
    for (int gi = tid; gi < H / 64; gi += kFThreads) {   // 64 columns = 8 permuted 16-byte entries
        float sx = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 q = reinterpret_cast<const uint4*>(xperm)[gi * 8 + i];
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) sx += __uint_as_float(u[j] << 16) + __uint_as_float(u[j] & 0xFFFF0000u);
        }
        xsum[gi] = sx;
    }
    __syncthreads();

    // ---------------------------------------------------------------- weight loads (routed: after the top-k)
    // called by all 32 lanes of warp 0: lane b issues box b, lanes 16.. the rest
    auto issue_loads = [&](int e) {
        const bool sh = (e >= E);
        const CUtensorMap* MG = sh ? &msg : &mg;
        const CUtensorMap* MU = sh ? &msu : &mu;
        const CUtensorMap* MD = sh ? &msd : &md;
        const int grow = (sh ? 0 : e * I) + rank * RG;
        const int drow = (sh ? 0 : e * H) + rank * RD;
        const uint32_t gsz = RG * (H / 64) * 2, dsz = RD * (I / 64) * 2;
        const size_t go = (size_t)grow * (H / 64), dO = (size_t)drow * (I / 64);
        if (lane < nbox_gu) {
            const int b = lane;
            mbar_arrive_expect_tx(&bar_gu[b], 2u * RG * 128 + (b == 0 ? 4 * gsz : 0));
            tma_load_2d(gcodes + (size_t)b * RG * 128, MG, b * 32, grow, &bar_gu[b]);
            tma_load_2d(ucodes + (size_t)b * RG * 128, MU, b * 32, grow, &bar_gu[b]);
            if (b == 0) {
                bulk_load(gsb, (sh ? a.sgs : a.gs) + go, gsz, &bar_gu[0]);
                bulk_load(gsb + RG * (H / 64), (sh ? a.sgb : a.gb) + go, gsz, &bar_gu[0]);
                bulk_load(usb, (sh ? a.sus : a.us) + go, gsz, &bar_gu[0]);
                bulk_load(usb + RG * (H / 64), (sh ? a.sub : a.ub) + go, gsz, &bar_gu[0]);
            }
        }
        if (lane == 31) {
            mbar_arrive_expect_tx(bar_dn, (uint32_t)RD * (I / 2) + 2 * dsz);
            for (int b = 0; b < nbox_dn; ++b) tma_load_2d(dcodes + (size_t)b * RD * 128, MD, b * 32, drow, bar_dn);
            bulk_load(dsb, (sh ? a.sds : a.ds) + dO, dsz, bar_dn);
            bulk_load(dsb + RD * (I / 64), (sh ? a.sdb : a.db) + dO, dsz, bar_dn);
        }
    };

    // ---------------------------------------------------------------- 1. router partial sums
    if (tid < 2 * E) {
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) sum = fmaf(rx[j], rw[j], sum);
        (tid / E ? logits : part)[r_e] = sum;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kFThreads) part[e] += logits[e];
    __syncthreads();
    // the shared expert needs no routing: its loads start once this CTA's router
    // reads are done, so that they do not delay the exchange everyone waits on
    if (shared_cluster && warp == 0) issue_loads(E);
    cluster_sync();
    {   // cluster sum of the partials, ranks in order; CTA r reduces experts [r*E/kCS, (r+1)*E/kCS)
        const int e0 = rank * E / kCS, e1 = (rank + 1) * E / kCS;
        for (int e = e0 + tid; e < e1; e += kFThreads) {
            float v[kCS];
#pragma unroll
            for (int r = 0; r < kCS; ++r) v[r] = ld_dsmem_f32(part + e, r);
            float s = 0.f;
#pragma unroll
            for (int r = 0; r < kCS; ++r) s += v[r];
            a.cpart[(size_t)slot * E + e] = s;
        }
        __syncthreads();
        if (tid == 0) atomic_add_release_gpu(&a.ctrl->decode_counter, 1u);
    }
    cluster_sync();   // every peer has read this CTA's partials; the buffers may be reused
    if (shared_cluster) {   // the shared cluster's gate sigmoid(x . g), all threads
        float d = 0.f;
        for (int h = tid * 8; h < H; h += kFThreads * 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(a.x + h);
            const float4 g0 = *reinterpret_cast<const float4*>(a.shared_gate + h);
            const float4 g1 = *reinterpret_cast<const float4*>(a.shared_gate + h + 4);
            const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                d = fmaf(__uint_as_float(u[j] << 16), gg[2 * j], d);
                d = fmaf(__uint_as_float(u[j] & 0xFFFF0000u), gg[2 * j + 1], d);
            }
        }
        d = warp_sum(d);
        if (lane == 0) gsum[warp] = d;   // gsum is free until the gate/up GEMV
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < kFWarps; ++w) t += gsum[w];
            *sel_w = 1.0f / (1.0f + expf(-t));
            *sel_e = E;
            if (rank == 0) *a.gamma_out = *sel_w;
        }
    }
    if (!shared_cluster) {
        // ------------------------------------------------------------ 1b. exchange, top-k
        if (tid == 0) {
            const uint64_t t0 = globaltimer();
            while (ld_acquire_u32(&a.ctrl->decode_counter) < (uint32_t)NG) {
                __nanosleep(20);
                if (globaltimer() - t0 > kWaitLimitNs) {
                    raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
        }
        __syncthreads();
        if (!*abort_flag) {
            for (int e = tid; e < E; e += kFThreads) {
                float v[kMaxSlots];
#pragma unroll
                for (int j = 0; j < kMaxSlots; ++j) v[j] = (j < NC) ? __ldcg(a.cpart + (size_t)j * E + e) : 0.f;
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxSlots; ++j) s += v[j];
                logits[e] = s + (a.router_bias ? a.router_bias[e] : 0.f);
            }
            __syncthreads();
            {
                __shared__ int32_t idx_s[8];
                __shared__ float v_s[8];
                __shared__ __align__(16) uint32_t cand[128];
                select_topk_block(logits, E, k, idx_s, v_s, cand);
                __syncthreads();
                if (warp == 0) {   // softmax over the selection (v_s[0] is the largest), one lane per slot
                    const float ex = lane < k ? expf(v_s[lane] - v_s[0]) : 0.f;
                    const float z = warp_sum(ex);
                    if (lane < k) {
                        const float w = ex / z;
                        if (lane == slot) { *sel_e = idx_s[lane]; *sel_w = w; }
                        if (G == 0) { a.idx_out[lane] = idx_s[lane]; a.w_out[lane] = w; }
                    }
                }
            }
            __syncthreads();
            if (warp == 0) {
                const int e = *sel_e;
                if (e < 0 || e >= E) { if (lane == 0) { raise_status(status, MOE_W4_STATUS_BAD_INDEX); *abort_flag = 1; } }
                else issue_loads(e);
            }
        }
    }
    __syncthreads();
    const bool run = !*abort_flag;

    // ---------------------------------------------------------------- 3. gate/up GEMV
    // 2*RG/16 row tiles (gate, then up) x KS splits of the 64-column groups
    if (run && mbar_wait(&bar_gu[0], 0, abort_flag, status)) {   // box 0 also carries the scales/biases
        const int ntile = 2 * (RG / 16), KS = kFWarps / ntile > 0 ? kFWarps / ntile : 1, ngrp = H / 64;
        for (int task = warp; task < ntile * KS; task += kFWarps) {
            const int t = task / KS, ks = task % KS;
            const bool up = t >= ntile / 2;
            const int r0 = (up ? t - ntile / 2 : t) * 16;
            const uint16_t* sb = up ? usb : gsb;
            float acc0 = 0.f, acc1 = 0.f;
            w4_gemv16<false>(up ? ucodes : gcodes, RG, r0, ks * ngrp / KS, (ks + 1) * ngrp / KS,
                             reinterpret_cast<const uint4*>(xperm), xsum, sb, sb + RG * (H / 64), H / 64, acc0,
                             acc1, bar_gu, abort_flag, status);
            if ((lane & 3) == 0) {
                red[task * 16 + (lane >> 2)] = acc0;
                red[task * 16 + (lane >> 2) + 8] = acc1;
            }
        }
        __syncthreads();
        for (int i = tid; i < 2 * RG; i += kFThreads) {   // sum the K splits in order
            const int t = i / 16, r = i % 16;
            float v = 0.f;
            for (int ks = 0; ks < KS; ++ks) v += red[(t * KS + ks) * 16 + r];
            (t < ntile / 2 ? gsum : usum)[(t % (ntile / 2)) * 16 + r] = v;
        }
    }
    __syncthreads();
    if (run)
        for (int i = tid; i < RG; i += kFThreads) hloc[i] = silu_f(gsum[i]) * usum[i];
    // ---------------------------------------------------------------- 4. exchange h inside the cluster
    cluster_sync();
    if (run) {
        // fp16 B fragments of h, permuted like x, and per-64-column sums
        for (int i = tid; i < I / 8; i += kFThreads) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = i * 8 + j;
                v[j] = ld_dsmem_f32(hloc + (col % RG), col / RG);
            }
            const uint32_t q0 = h2_as_u32(__floats2half2_rn(v[0], v[4])), q1 = h2_as_u32(__floats2half2_rn(v[1], v[5]));
            const uint32_t q2 = h2_as_u32(__floats2half2_rn(v[2], v[6])), q3 = h2_as_u32(__floats2half2_rn(v[3], v[7]));
            reinterpret_cast<uint4*>(hperm)[i] = make_uint4(q0, q1, q2, q3);
        }
    }
    cluster_sync();   // peers may leave once everyone has read their h
    if (run) {
        for (int gi = tid; gi < I / 64; gi += kFThreads) {
            float s = 0.f;
            for (int i = gi * 8; i < gi * 8 + 8; ++i) {
                const uint4 q = reinterpret_cast<const uint4*>(hperm)[i];
                const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(u32_as_h2(u[j]));
                    s += f.x + f.y;
                }
            }
            hsum[gi] = s;
        }
    }
    __syncthreads();
    // ---------------------------------------------------------------- 5. down GEMV
    if (run && mbar_wait(bar_dn, 0, abort_flag, status)) {
        const int ntile = RD / 16;
        const float wsel = *sel_w;
        for (int t = warp; t < ntile; t += kFWarps) {
            float acc0 = 0.f, acc1 = 0.f;
            w4_gemv16<true>(dcodes, RD, t * 16, 0, I / 64, reinterpret_cast<const uint4*>(hperm), hsum, dsb,
                            dsb + RD * (I / 64), I / 64, acc0, acc1, nullptr, abort_flag, status);
            if ((lane & 3) == 0) {
                const int o = rank * RD + t * 16 + (lane >> 2);
                a.ybuf[(size_t)slot * H + o] = acc0 * wsel;
                a.ybuf[(size_t)slot * H + o + 8] = acc1 * wsel;
            }
        }
    }
    // ---------------------------------------------------------------- 6. combine: last of the k+1 CTAs per row block
    __syncthreads();
    if (tid == 0) *last_flag = (atomic_add_acq_rel_gpu(&a.ctrl->pad[rank], 1u) == (unsigned)(NC - 1));
    __syncthreads();
    if (*last_flag) {
        for (int o = rank * RD + tid; o < (rank + 1) * RD; o += kFThreads) {
            float v[kMaxSlots];
#pragma unroll
            for (int j = 0; j < kMaxSlots; ++j) v[j] = (j < NC) ? __ldcg(a.ybuf + (size_t)j * H + o) : 0.f;
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxSlots; ++j) s += v[j];
            a.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
        }
        __syncthreads();
        if (tid == 0) {
            a.ctrl->pad[rank] = 0;
            // the last row block to finish resets the exchange counter for the next call
            if (atomicAdd(&a.ctrl->pad[kCS], 1u) == (unsigned)(kCS - 1)) {
                a.ctrl->decode_counter = 0;
                a.ctrl->pad[kCS] = 0;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn2)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn2 encode_fn2() {
    static EncodeTiledFn2 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn2>(p);
    }
    return fn;
}

// codes [rows][cols/8] uint32, box = 32 words x box_rows, 128-byte swizzle
static bool codes_map(CUtensorMap* m, const uint32_t* codes, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn2 fn = encode_fn2();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols / 8, rows};
    const cuuint64_t strides[1] = {cols / 8 * 4};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decode_fused_supported(const moe_w4_layer& L) {
    if (L.H % 256 || L.I % 256 || L.H / kCS > 256 || L.I / kCS > 256) return false;
    if ((L.I / kCS) % 16 || (L.H / kCS) % 16 || L.H / 256 > 16) return false;
    if (L.E < 128 || L.E > 256 || L.E % 32) return false;   // top-k: E/32 warps sort 32 scores each; 2E floats of partials
    if (L.H > 64 * kCS * (L.top_k + 1)) return false;   // <= 64 router rows per CTA (32 per thread)
    const FusedSmem s(L.H, L.E, L.I);
    return s.total + 1024 + 256 <= 227 * 1024;   // + static shared memory of the kernel
}

size_t decode_fused_scratch(const moe_w4_layer& L) {
    return ((size_t)(L.top_k + 1) * L.E + (size_t)(L.top_k + 1) * L.H) * 4;
}

cudaError_t launch_decode_fused(const moe_w4_layer& L, const uint16_t* x, uint16_t* out, const DecodeWs& d,
                                cudaStream_t st) {
    const int H = L.H, E = L.E, I = L.I, k = L.top_k;
    const int RG = I / kCS, RD = H / kCS;
    CUtensorMap mg, mu, md, msg, msu, msd;
    bool ok = codes_map(&mg, L.gate.codes, (uint64_t)E * I, H, RG) && codes_map(&mu, L.up.codes, (uint64_t)E * I, H, RG) &&
              codes_map(&md, L.down.codes, (uint64_t)E * H, I, RD) && codes_map(&msg, L.sh_gate.codes, I, H, RG) &&
              codes_map(&msu, L.sh_up.codes, I, H, RG) && codes_map(&msd, L.sh_down.codes, H, I, RD);
    if (!ok) return cudaErrorInvalidValue;
    FusedArgs a{};
    a.x = x; a.router_w = L.router_w; a.router_bias = L.router_bias; a.shared_gate = L.shared_gate;
    a.gs = L.gate.scales; a.gb = L.gate.biases; a.us = L.up.scales; a.ub = L.up.biases;
    a.ds = L.down.scales; a.db = L.down.biases;
    a.sgs = L.sh_gate.scales; a.sgb = L.sh_gate.biases; a.sus = L.sh_up.scales; a.sub = L.sh_up.biases;
    a.sds = L.sh_down.scales; a.sdb = L.sh_down.biases;
    a.cpart = d.fused_cpart; a.ybuf = d.fused_ybuf;
    a.idx_out = d.idx; a.w_out = d.w; a.gamma_out = d.gamma; a.out = out;
    a.ctrl = d.ctrl;
    a.H = H; a.E = E; a.I = I; a.k = k;
    const FusedSmem s(H, E, I);
    const size_t smem = s.total + 1024;
    static size_t attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev] < smem) {   // dynamic + static shared memory must stay within the opt-in limit
        const cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((k + 1) * kCS);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_fused_kernel, a, mg, mu, md, msg, msu, msd);
}

}  // namespace mw4
