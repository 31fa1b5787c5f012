// Fused batch-1 decode: the whole layer for one token in one launch.
// ("Optimizing on-device inference for Apple Silicon", sections "Optimise the
// single-row weight path" -- groups of threads cooperate on outputs while
// reading different parts of the weight matrix -- and "Reduce intermediate
// state and traffic" -- gate/up projections fused with the gated activation,
// the output projection fused with the routing scores and the shared expert.)
//
// Grid: (k+1) experts x 16 CTAs, in clusters of 4 (one CTA per SM; the host
// checks that every cluster fits on the GPU at once).  Expert slot j < k is
// the j-th selected expert, slot k the shared expert.  CTA i (0..15) of an
// expert owns gate/up rows [i*I/16, (i+1)*I/16) and down rows
// [i*H/16, (i+1)*H/16) of it.
//
//   1. router: every CTA sums x . W_r over its own 1/(16 (k+1)) slice of the H
//      rows for all E experts (these loads go out first); the 4 slices of a
//      cluster are added through distributed shared memory, the cluster sums
//      are published in global memory and, once all are in (bounded wait: all
//      CTAs are co-resident), every routed CTA adds them in a fixed order and
//      selects the top-k.  Every value that crosses CTAs through global memory
//      is an 8-byte (value, call tag) word, so that a reader waits on the data
//      itself rather than on a counter and then the data.  The shared expert does not wait for the routing: it
//      starts loading its weights as soon as its own router reads are done.
//   2. TMA loads the CTA's slices of the packed codes (128-byte swizzle) and
//      its scales/biases; the gate/up slices are consumed box by box as they
//      land.
//   3. gate/up GEMV on the tensor cores as a dot-product engine: mma.sync
//      m16n8k16 with fp16 A = 1024 + q (even nibbles) or 1024 + 16 q (odd
//      nibbles), one bitwise op per pair, and B = x in fp16 with the odd
//      positions divided by 16; fp32 accumulation per 64-column group, then
//      s*(acc - 1024*sum(B)) + b*sum(x).  SwiGLU in fp32.  The instances for
//      one-byte codes take 1024 + q (8-bit codes) or the exact E4M3 value (no
//      offset) for bytes (0, 2) and (1, 3) of a word, with B in matching
//      4-column units and no division by 16.
//   4. h: every CTA publishes its slice of h in global memory; the 16 CTAs of
//      an expert wait (bounded) until all 16 slices carry the tag and read all of h.
//   5. down GEMV the same way with h in fp16, scaled by the routing weight
//      (or the shared gate), written per expert.
//   6. per block of output rows, the shared expert's CTA (it needs no routing,
//      so it is usually done first) waits (bounded) for the k routed outputs,
//      adds the k+1 in slot order and writes bf16 out.
// No step waits on another CTA except these bounded exchanges and the hardware
// cluster barriers.
#include "common.cuh"
#include "internal.h"

namespace mw4 {

constexpr int kCS = 4;                                   // CTAs per cluster
constexpr int kPE = kCS * kFusedClustersPerExpert;       // CTAs per expert (16)
constexpr int kFThreads = 512;                           // 16 warps
constexpr int kFWarps = kFThreads / 32;
constexpr int kMaxSlots = 9;                             // k + 1 <= 9

struct FusedArgs {
    const uint16_t* x;          // [H] bf16
    const float* router_w;      // [H][E]
    const float* router_bias;   // [E] or NULL
    const float* shared_gate;   // [H]
    const uint16_t* gs; const uint16_t* gb; const uint16_t* us; const uint16_t* ub;   // routed gate/up s, b
    const uint16_t* ds; const uint16_t* db;                                             // routed down s, b
    const uint16_t* sgs; const uint16_t* sgb; const uint16_t* sus; const uint16_t* sub; // shared
    const uint16_t* sds; const uint16_t* sdb;
    uint64_t* cpart;            // [4(k+1)][E] cluster partial scores, tagged with the call
    uint64_t* hx;               // [k+1][I] h of every expert, tagged with the call
    uint64_t* ybuf;             // [k+1][H] weighted expert outputs, tagged with the call
    int32_t* idx_out;           // [k] (for inspection)
    float* w_out;               // [k]
    float* gamma_out;           // [1]
    uint16_t* out;              // [H] bf16
    Ctrl* ctrl;
    int H, E, I, k;
};

// smem carve-up (byte offsets from a 1024-aligned base), computed on both sides
struct FusedSmem {
    uint32_t gcodes, ucodes, dcodes, gsb, usb, dsb, xperm, xsum, xbs, part, logits, gsum, usum, hperm, hsum,
        hbs, red, misc, total;
    int RG, RD;
    __host__ __device__ FusedSmem(int H, int E, int I, int bits) {
        RG = I / kPE;
        RD = H / kPE;
        uint32_t o = 0;
        auto take = [&](uint32_t bytes, uint32_t align) {
            o = (o + align - 1) / align * align;
            const uint32_t at = o;
            o += bytes;
            return at;
        };
        gcodes = take(RG * H / 8 * bits, 1024);
        ucodes = take(RG * H / 8 * bits, 1024);
        dcodes = take(RD * I / 8 * bits, 1024);
        gsb = take(2 * RG * (H / 64) * 2, 16);   // scales then biases
        usb = take(2 * RG * (H / 64) * 2, 16);
        dsb = take(2 * RD * (I / 64) * 2, 16);
        xperm = take(H * 2, 16);
        xsum = take(H / 64 * 4, 16);
        xbs = take(H / 64 * 4, 16);
        part = take(E * 4, 16);
        logits = take(E * 4, 16);
        gsum = take(RG * 4, 16);
        usum = take(RG * 4, 16);
        hperm = take(I * 2, 16);
        hsum = take(I / 64 * 4, 16);
        hbs = take(I / 64 * 4, 16);
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
// The two halves of cluster_sync, for work in between.
MW4_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
MW4_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
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

// One warp: rows [r0, r0+16) of a swizzled codes tile set, one 64-column
// group; adds the group's dot products of rows r0+g and r0+g+8 (g = lane/4)
// to d[0] and d[2].  A holds fp16 1024 + q for the even nibbles of a code
// byte and 1024 + 16 q for the odd ones (one bitwise op per pair, one shift
// per word); B (`bperm`, 16 bytes per (32-column block, lane%4)) holds the
// matching activations, the odd positions divided by 16, so that every
// product is q * value + 1024 * (stored B value).
MW4_DEV void w4_group_mma(const uint8_t* codes, int rows, int r0, int grp, const uint4* bperm, float (&d)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    constexpr uint32_t M = 0x64006400u;
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
        a[0] = (wg & 0x000F000Fu) | M;   // nibbles 0, 4
        a[1] = (wh & 0x000F000Fu) | M;
        a[2] = (wg & 0x00F000F0u) | M;   // nibbles 1, 5 (x16)
        a[3] = (wh & 0x00F000F0u) | M;
        mma_f16_16816(d, a, bv.x, bv.y);
        const uint32_t wg8 = wg >> 8, wh8 = wh >> 8;
        a[0] = (wg8 & 0x000F000Fu) | M;  // nibbles 2, 6
        a[1] = (wh8 & 0x000F000Fu) | M;
        a[2] = (wg8 & 0x00F000F0u) | M;  // nibbles 3, 7 (x16)
        a[3] = (wh8 & 0x00F000F0u) | M;
        mma_f16_16816(d, a, bv.z, bv.w);
    }
}

// Code formats of the one-kernel decode: unsigned 4-bit, unsigned 8-bit, FP8 E4M3.
enum : int { kCodeU4 = 0, kCodeU8 = 1, kCodeE4M3 = 2 };

// One warp, one-byte codes: rows [r0, r0+16), one 64-column group = 4 chunks of
// 16 codes (one 16-byte chunk of 4 words per row, one MMA each); adds the
// group's dot products of rows r0+g and r0+g+8 to d[0] and d[2].  Lane c takes
// word c of a chunk: 8-bit codes give fp16 1024 + q for bytes (0, 2) and (1, 3)
// (one bitwise op per pair, one shift per word), E4M3 codes their exact values;
// B (`bperm`, 8 bytes per 4-column unit u = chunk * 4 + lane%4) holds the
// matching activations (x[4u], x[4u+2]), (x[4u+1], x[4u+3]).
template <bool E4M3>
MW4_DEV void w8_group_mma(const uint8_t* codes, int rows, int r0, int grp, const uint2* bperm, float (&d)[4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    constexpr uint32_t M = 0x64006400u;
    // both rows of the thread share the swizzle phase g; the group's 4 chunks lie
    // inside one box of 8 chunks
    const int ch0 = grp * 4;
    const uint8_t* row0 = codes + (size_t)(ch0 >> 3) * rows * 128 + (r0 + g) * 128 + c * 4;
    const uint8_t* row1 = row0 + 8 * 128;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int ch = ch0 + h;
        const int off = ((ch & 7) ^ g) << 4;
        const uint32_t wg = *reinterpret_cast<const uint32_t*>(row0 + off);
        const uint32_t wh = *reinterpret_cast<const uint32_t*>(row1 + off);
        const uint2 bv = bperm[ch * 4 + c];
        uint32_t a[4];
        if (E4M3) {
            e4m3x4_to_f16(wg, a[0], a[2]);   // (c0, c2), (c1, c3)
            e4m3x4_to_f16(wh, a[1], a[3]);
        } else {
            a[0] = (wg & 0x00FF00FFu) | M;   // bytes 0, 2
            a[1] = (wh & 0x00FF00FFu) | M;
            a[2] = ((wg >> 8) & 0x00FF00FFu) | M;   // bytes 1, 3
            a[3] = ((wh >> 8) & 0x00FF00FFu) | M;
        }
        mma_f16_16816(d, a, bv.x, bv.y);
    }
}

// Rows r0+g and r0+g+8 dotted with the activation over groups [grp0, grp1):
// per group w = s*q + b, so the dot is s * (sum of q*value) + b * (sum of
// values); `bsum` holds per-group sums of the stored B values (for the 1024
// offset), `tsum` the true sums of the activation.
// With one-byte codes a TMA box holds 2 groups (128 columns) instead of 4, and
// `bperm` is read as 8-byte units.
template <int CODE>
MW4_DEV bool w4_gemv16(const uint8_t* codes, int rows, int r0, int grp0, int grp1, const uint4* bperm,
                       const float* bsum, const float* tsum, const uint16_t* sc, const uint16_t* bi, int ngrp_row,
                       float& acc0, float& acc1, uint64_t* box_bars, volatile int* abort_flag, unsigned int* status) {
    const int lane = threadIdx.x & 31, g = lane >> 2;
    constexpr int kIn = 4;   // groups in flight: independent MMA chains
    constexpr int kGpb = CODE == kCodeU4 ? 4 : 2;   // groups per TMA box
    for (int grp = grp0; grp < grp1; grp += kIn) {
        if (box_bars) {
            for (int q = 0; q < kIn; ++q)
                if (grp + q < grp1 && ((grp + q) % kGpb) == 0 || (q == 0 && grp + q < grp1))
                    if (!mbar_wait(&box_bars[(grp + q) / kGpb], 0, abort_flag, status)) return false;
        }
        float d[kIn][4];
#pragma unroll
        for (int q = 0; q < kIn; ++q) {
            d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.f;
            if (grp + q < grp1) {
                if (CODE == kCodeU4)
                    w4_group_mma(codes, rows, r0, grp + q, bperm, d[q]);
                else
                    w8_group_mma<CODE == kCodeE4M3>(codes, rows, r0, grp + q, reinterpret_cast<const uint2*>(bperm),
                                                    d[q]);
            }
        }
        // every lane of a row group holds the same column sums (B is the same for all n)
#pragma unroll
        for (int q = 0; q < kIn; ++q) {
            const int gg = grp + q;
            if (gg >= grp1) break;
            const float bs = bsum[gg], xs = tsum[gg];
            const float s0 = bf16_bits_to_float(sc[(r0 + g) * ngrp_row + gg]);
            const float b0 = bf16_bits_to_float(bi[(r0 + g) * ngrp_row + gg]);
            const float s1 = bf16_bits_to_float(sc[(r0 + g + 8) * ngrp_row + gg]);
            const float b1 = bf16_bits_to_float(bi[(r0 + g + 8) * ngrp_row + gg]);
            acc0 = fmaf(s0, d[q][0] - 1024.f * bs, fmaf(b0, xs, acc0));
            acc1 = fmaf(s1, d[q][2] - 1024.f * bs, fmaf(b1, xs, acc1));
        }
    }
    return true;
}

// Shape parameters given at compile time (kH, kI, kE, kK non-zero) fold the
// GEMVs' shared-memory address arithmetic into constants: measured 1.6x faster
// for the dot-product loops than the same code with run-time strides.  The
// instance with all four zero takes every shape from the arguments.
template <int kH, int kI, int kE, int kK, int CODE>
__global__ void __launch_bounds__(kFThreads, 1)
decode_fused_kernel(const __grid_constant__ FusedArgs a, const __grid_constant__ CUtensorMap mg,
                    const __grid_constant__ CUtensorMap mu, const __grid_constant__ CUtensorMap md,
                    const __grid_constant__ CUtensorMap msg, const __grid_constant__ CUtensorMap msu,
                    const __grid_constant__ CUtensorMap msd) {
    const int H = kH ? kH : a.H, E = kE ? kE : a.E, I = kI ? kI : a.I, k = kK ? kK : a.k;
    constexpr int kBits = CODE == kCodeU4 ? 4 : 8;
    const FusedSmem L(H, E, I, kBits);
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
    float* xbs = reinterpret_cast<float*>(sm + L.xbs);
    float* part = reinterpret_cast<float*>(sm + L.part);
    float* logits = reinterpret_cast<float*>(sm + L.logits);
    float* gsum = reinterpret_cast<float*>(sm + L.gsum);
    float* usum = reinterpret_cast<float*>(sm + L.usum);
    uint32_t* hperm = reinterpret_cast<uint32_t*>(sm + L.hperm);
    float* hsum = reinterpret_cast<float*>(sm + L.hsum);
    float* hbs = reinterpret_cast<float*>(sm + L.hbs);
    float* red = reinterpret_cast<float*>(sm + L.red);
    uint8_t* misc = sm + L.misc;
    // TMA boxes of 128-byte code rows: 256 columns of 4-bit codes, 128 of one-byte codes
    const int nbox_gu = H * kBits / 1024, nbox_dn = I * kBits / 1024 > 0 ? I * kBits / 1024 : 1;
    uint64_t* bar_gu = reinterpret_cast<uint64_t*>(misc);               // [nbox_gu] (<= 16)
    uint64_t* bar_dn = bar_gu + 16;                                      // [1]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_dn + 1);
    int* sel_e = reinterpret_cast<int*>(bar_dn + 2);                     // selected expert of this cluster
    float* sel_w = reinterpret_cast<float*>(sel_e + 1);                  // its weight (or gamma)
    uint32_t* xtag_s = reinterpret_cast<uint32_t*>(sel_e + 3);            // this call's exchange tag
    uint32_t* xinj_s = reinterpret_cast<uint32_t*>(sel_e + 4);            // test hook: skip a publish

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // clusters are consecutive blocks: expert slot = block / kPE, CTA ei of the
    // expert = block % kPE; cluster cid, rank inside the cluster for DSMEM
    const int rank = (int)cluster_rank(), cid = (int)cluster_id();
    const int G = blockIdx.x, slot = G / kPE, ei = G % kPE;
    const int NC = k + 1, NG = NC * kPE, NCL = NC * kFusedClustersPerExpert;
    const bool shared_cluster = (slot == k);
    unsigned int* status = &a.ctrl->status;

    // The kernel may start before the previous kernel on the stream has finished
    // (programmatic dependent launch): until griddep_wait() it touches only
    // weights, its own shared memory and the tensor maps.
    // The router's loads go out first: thread (e, half) sums half of this CTA's
    // slice of the H rows for expert e; its W_r column slice is requested before
    // the wait, the matching x values (the same for the whole warp) after it.
    const int rh0 = (int)((long)G * H / NG), rh1 = (int)((long)(G + 1) * H / NG);
    const int rnh = rh1 - rh0, rhalf = rnh / 2;
    const int r_e = tid % E, r_hb = (tid / E) ? rhalf : 0, r_he = (tid / E) ? rnh : rhalf;
    float rw[32], rx[32];
    if (tid < 2 * E) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const bool in = r_hb + j < r_he;
            rw[j] = in ? __ldg(a.router_w + (size_t)(rh0 + r_hb + j) * E + r_e) : 0.f;
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
    griddep_wait();   // from here on: x, the workspace and its counters
    // Values crossing CTAs carry this call's tag (the call counter + 1): a reader
    // polls the data itself instead of a counter and then the data.  CTA 0 advances
    // the counter once every cluster's router sum carries the tag, i.e. once every
    // CTA has read it.
    if (tid == 0) {
        *xtag_s = ld_acquire_u32(&a.ctrl->pad[kCtrlEpochWord]) + 1u;
        *xinj_s = ld_acquire_u32(&a.ctrl->pad[kCtrlInjectWord]);
    }
    if (tid < 2 * E) {
#pragma unroll
        for (int j = 0; j < 32; ++j) rx[j] = (r_hb + j < r_he) ? bf16_bits_to_float(__ldg(a.x + rh0 + r_hb + j)) : 0.f;
    }

    // ---------------------------------------------------------------- weight loads (routed: after the top-k)
    // called by all 32 lanes of warp 0
    auto issue_loads = [&](int e) {
        const bool sh = (e >= E);
        const CUtensorMap* MG = sh ? &msg : &mg;
        const CUtensorMap* MU = sh ? &msu : &mu;
        const CUtensorMap* MD = sh ? &msd : &md;
        const int grow = (sh ? 0 : e * I) + ei * RG;
        const int drow = (sh ? 0 : e * H) + ei * RD;
        const uint32_t gsz = RG * (H / 64) * 2, dsz = RD * (I / 64) * 2;
        const size_t go = (size_t)grow * (H / 64), dO = (size_t)drow * (I / 64);
        // in the order the GEMVs consume them: the gate/up scales and biases (box 0's
        // barrier waits for them too), then gate and up of box 0, of box 1, ..., then down
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar_gu[0], 2u * RG * 128 + 4 * gsz);
            bulk_load(gsb, (sh ? a.sgs : a.gs) + go, gsz, &bar_gu[0]);
            bulk_load(gsb + RG * (H / 64), (sh ? a.sgb : a.gb) + go, gsz, &bar_gu[0]);
            bulk_load(usb, (sh ? a.sus : a.us) + go, gsz, &bar_gu[0]);
            bulk_load(usb + RG * (H / 64), (sh ? a.sub : a.ub) + go, gsz, &bar_gu[0]);
        }
        __syncwarp();
        for (int p = lane; p < 2 * nbox_gu; p += 32) {   // p = 2 box + matrix
            const int b = p >> 1;
            if ((p & 1) == 0 && b != 0) mbar_arrive_expect_tx(&bar_gu[b], 2u * RG * 128);
            __syncwarp(__activemask());
            tma_load_2d(((p & 1) ? ucodes : gcodes) + (size_t)b * RG * 128, (p & 1) ? MU : MG, b * 32, grow,
                        &bar_gu[b]);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_dn, (uint32_t)RD * (I * kBits / 8) + 2 * dsz);
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
            if (!(*xinj_s != 0u && cid == 0)) st_tagged(a.cpart + (size_t)cid * E + e, s, *xtag_s);
        }
    }
    // the shared expert needs no routing: its loads start once its router sums are
    // published, so that issuing them does not delay the exchange everyone waits on
    if (shared_cluster && warp == 0) issue_loads(E);
    // this CTA has read its peers' partials; the matching wait (every peer has read
    // this CTA's, so the buffer may be reused) comes before the gate/up GEMV reuses it
    cluster_arrive();
    // x for the GEMVs is prepared here, off the router's critical path, while the
    // other CTAs' router sums come in
    // x as fp16 B fragments, one thread per 16-byte entry: for 4-bit codes
    // entry i (32-column block i/4, lane%4 = i%4) holds {x[8i], x[8i+4]},
    // {x[8i+1], x[8i+5]}/16, {x[8i+2], x[8i+6]}, {x[8i+3], x[8i+7]}/16; for
    // one-byte codes {x[8i], x[8i+2]}, {x[8i+1], x[8i+3]}, {x[8i+4], x[8i+6]},
    // {x[8i+5], x[8i+7]} (the 4-column units 2i and 2i+1); plus the per-64-column group
    // sums of the stored values (xbs) and of the values the products use
    // (xsum), reduced over the 8 lanes of a group (H/8 is a multiple of 32, so
    // the loop runs whole warps)
    for (int i = tid; i < H / 8; i += kFThreads) {
        const uint4 v = *reinterpret_cast<const uint4*>(a.x + i * 8);
        const uint32_t e[4] = {v.x, v.y, v.z, v.w};   // pairs (0,1) (2,3) (4,5) (6,7)
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(e[j] << 16);
            f[2 * j + 1] = __uint_as_float(e[j] & 0xFFFF0000u);
        }
        float sb = 0.f, so = 0.f;   // sums of the stored even / odd entries
        bool bad = false;
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            bad |= !(fabsf(f[j]) <= 65504.f) || !(fabsf(f[j + 4]) <= 65504.f);
            __half2 h2;
            if (CODE == kCodeU4) {
                const float m = (j & 1) ? 0.0625f : 1.0f;
                h2 = __floats2half2_rn(f[j] * m, f[j + 4] * m);
            } else {   // 4-column units (x[4u], x[4u+2]), (x[4u+1], x[4u+3])
                const int b = (j >> 1) * 4 + (j & 1);
                h2 = __floats2half2_rn(f[b], f[b + 2]);
            }
            q[j] = h2_as_u32(h2);
            const float2 back = __half22float2(h2);
            if (CODE == kCodeU4 && (j & 1)) so += back.x + back.y; else sb += back.x + back.y;
        }
        reinterpret_cast<uint4*>(xperm)[i] = make_uint4(q[0], q[1], q[2], q[3]);
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) {
            sb += __shfl_xor_sync(0xffffffffu, sb, off);
            so += __shfl_xor_sync(0xffffffffu, so, off);
        }
        if ((i & 7) == 0) {   // E4M3 products carry no 1024 offset
            xbs[i / 8] = CODE == kCodeE4M3 ? 0.f : sb + so;
            xsum[i / 8] = sb + 16.f * so;
        }
        if (bad) raise_status(status, MOE_W4_STATUS_FP16_RANGE);
    }
    __syncthreads();
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
            if (ei == 0) *a.gamma_out = *sel_w;
        }
    }
    if (!shared_cluster) {
        // ------------------------------------------------------------ 1b. exchange, top-k
        {
            const uint32_t xtag = *xtag_s;
            for (int e = tid; e < E; e += kFThreads) {   // cluster sums added in cluster order, all loads in flight
                constexpr int kMaxCl = kMaxSlots * kFusedClustersPerExpert;
                uint64_t v[kMaxCl];
#pragma unroll
                for (int j = 0; j < kMaxCl; ++j) v[j] = (j < NCL) ? ld_tagged(a.cpart + (size_t)j * E + e) : 0ull;
                // re-read the sums that do not carry this call's tag yet (bounded)
                const uint64_t t0 = globaltimer();
                while (true) {
                    bool all = true;
#pragma unroll
                    for (int j = 0; j < kMaxCl; ++j)
                        if (j < NCL && tag_of(v[j]) != xtag) {
                            all = false;
                            v[j] = ld_tagged(a.cpart + (size_t)j * E + e);
                        }
                    if (all) break;
                    if (globaltimer() - t0 > kWaitLimitNs) {
                        raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                }
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxCl; ++j) s += (j < NCL) ? val_of(v[j]) : 0.f;
                logits[e] = s + (a.router_bias ? a.router_bias[e] : 0.f);
            }
            __syncthreads();
            // every cluster's sum carries the tag, so every CTA has read the counter
            if (G == 0 && tid == 0 && !*abort_flag) a.ctrl->pad[kCtrlEpochWord] = xtag;
        }
        if (!*abort_flag) {
            // one warp selects, weighs and issues the loads of this CTA's expert
            if (warp == 0) {
                int sidx;
                float sval;
                warp_topk_sorted<8>(logits, E, k, sidx, sval);
                const int e = __shfl_sync(0xffffffffu, sidx, slot);
                // the loads first: the routing weight is needed only by the down GEMV
                if (e < 0 || e >= E) {
                    if (lane == 0) { raise_status(status, MOE_W4_STATUS_BAD_INDEX); *abort_flag = 1; }
                } else {
                    issue_loads(e);
                }
                const float v0 = __shfl_sync(0xffffffffu, sval, 0);   // the largest selected score
                const float ex = lane < k ? expf(sval - v0) : 0.f;
                const float z = warp_sum(ex);
                const float w = ex / z;   // softmax over the selection
                const float we = __shfl_sync(0xffffffffu, w, slot);
                if (lane == 0) { *sel_e = e; *sel_w = we; }
                if (G == 0 && lane < k) { a.idx_out[lane] = sidx; a.w_out[lane] = w; }
            }
        }
    }
    __syncthreads();
    const bool run = !*abort_flag;

    cluster_wait();   // every peer has read this CTA's partials: red (= part) may be written
    // ---------------------------------------------------------------- 3. gate/up GEMV
    // 2*RG/16 row tiles (gate, then up) x KS splits of the 64-column groups
    // box 0 also carries the scales/biases; the block agrees on the outcome of the wait
    const bool gu_ok = __syncthreads_and(run ? mbar_wait(&bar_gu[0], 0, abort_flag, status) : 0);
    if (gu_ok) {
        const int ntile = 2 * (RG / 16), KS = kFWarps / ntile > 0 ? kFWarps / ntile : 1, ngrp = H / 64;
        for (int task = warp; task < ntile * KS; task += kFWarps) {
            const int t = task / KS, ks = task % KS;
            const bool up = t >= ntile / 2;
            const int r0 = (up ? t - ntile / 2 : t) * 16;
            const uint16_t* sb = up ? usb : gsb;
            float acc0 = 0.f, acc1 = 0.f;
            // split ks takes its share of each half of the columns, so that every warp
            // starts on an early box and, once the last box lands, has one box left
            const int half = ngrp / 2;
            for (int hf = 0; hf < 2; ++hf)
                w4_gemv16<CODE>(up ? ucodes : gcodes, RG, r0, hf * half + ks * half / KS, hf * half + (ks + 1) * half / KS,
                          reinterpret_cast<const uint4*>(xperm), xbs, xsum, sb, sb + RG * (H / 64), H / 64, acc0, acc1,
                          bar_gu, abort_flag, status);
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
    // ---------------------------------------------------------------- 4. h through global memory
    // this CTA's slice of h, tagged; published even after an abort (as zeros), so
    // that no CTA of the expert waits in vain
    {
        const uint32_t xtag = *xtag_s;
        for (int i = tid; i < RG; i += kFThreads)
            st_tagged(a.hx + (size_t)slot * I + ei * RG + i, gu_ok ? silu_f(gsum[i]) * usum[i] : 0.f, xtag);
    }
    const bool h_in = gu_ok && !*abort_flag;
    if (h_in) {
        // fp16 B fragments of h, laid out like x, once all 16 slices carry this
        // call's tag
        const uint32_t xtag = *xtag_s;
        for (int i = tid; i < I / 8; i += kFThreads) {
            const uint64_t* src = a.hx + (size_t)slot * I + i * 8;
            uint64_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = ld_tagged(src + j);
            const uint64_t t0 = globaltimer();
            while (true) {
                bool all = true;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (tag_of(w[j]) != xtag) {
                        all = false;
                        w[j] = ld_tagged(src + j);
                    }
                if (all) break;
                if (globaltimer() - t0 > kWaitLimitNs) {
                    raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = val_of(w[j]);
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) bad |= !(fabsf(v[j]) <= 65504.f);
            if (bad) raise_status(status, MOE_W4_STATUS_FP16_RANGE);
            uint32_t q0, q1, q2, q3;
            if (CODE == kCodeU4) {
                q0 = h2_as_u32(__floats2half2_rn(v[0], v[4]));
                q1 = h2_as_u32(__floats2half2_rn(v[1] * 0.0625f, v[5] * 0.0625f));
                q2 = h2_as_u32(__floats2half2_rn(v[2], v[6]));
                q3 = h2_as_u32(__floats2half2_rn(v[3] * 0.0625f, v[7] * 0.0625f));
            } else {   // 4-column units, as for x
                q0 = h2_as_u32(__floats2half2_rn(v[0], v[2]));
                q1 = h2_as_u32(__floats2half2_rn(v[1], v[3]));
                q2 = h2_as_u32(__floats2half2_rn(v[4], v[6]));
                q3 = h2_as_u32(__floats2half2_rn(v[5], v[7]));
            }
            reinterpret_cast<uint4*>(hperm)[i] = make_uint4(q0, q1, q2, q3);
        }
    }
    __syncthreads();
    const bool h_ok = h_in && !*abort_flag;
    if (h_ok) {   // per-64-value group sums of h: one warp per group, lanes 0..7 one 8-value entry each
        for (int gi = warp; gi < I / 64; gi += kFWarps) {
            float sb = 0.f, so = 0.f;
            if (lane < 8) {
                const uint4 q = reinterpret_cast<const uint4*>(hperm)[gi * 8 + lane];
                const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __half22float2(u32_as_h2(u[j]));
                    if (CODE == kCodeU4 && (j & 1)) so += f.x + f.y; else sb += f.x + f.y;
                }
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                sb += __shfl_xor_sync(0xffffffffu, sb, off);
                so += __shfl_xor_sync(0xffffffffu, so, off);
            }
            if (lane == 0) {
                hbs[gi] = CODE == kCodeE4M3 ? 0.f : sb + so;   // E4M3 products carry no 1024 offset
                hsum[gi] = sb + 16.f * so;
            }
        }
    }
    // ---------------------------------------------------------------- 5. down GEMV
    griddep_launch_dependents();   // the next kernel on the stream may start its prologue
    // RD/16 row tiles x KS splits of the 64-column groups
    const bool dn_ok = __syncthreads_and(h_ok ? mbar_wait(bar_dn, 0, abort_flag, status) : 0);
    const uint32_t xtag = *xtag_s;
    if (dn_ok) {
        const int ntile = RD / 16, KS = kFWarps / ntile > 0 ? kFWarps / ntile : 1, ngrp = I / 64;
        for (int task = warp; task < ntile * KS; task += kFWarps) {
            const int t = task / KS, ks = task % KS;
            float acc0 = 0.f, acc1 = 0.f;
            w4_gemv16<CODE>(dcodes, RD, t * 16, ks * ngrp / KS, (ks + 1) * ngrp / KS, reinterpret_cast<const uint4*>(hperm),
                      hbs, hsum, dsb, dsb + RD * (I / 64), I / 64, acc0, acc1, nullptr, abort_flag, status);
            if ((lane & 3) == 0) {
                red[task * 16 + (lane >> 2)] = acc0;
                red[task * 16 + (lane >> 2) + 8] = acc1;
            }
        }
        __syncthreads();
        const float wsel = *sel_w;
        for (int i = tid; i < RD; i += kFThreads) {   // sum the K splits in order
            const int t = i / 16, r = i % 16;
            float v = 0.f;
            for (int ks = 0; ks < KS; ++ks) v += red[(t * KS + ks) * 16 + r];
            st_tagged(a.ybuf + (size_t)slot * H + ei * RD + i, v * wsel, xtag);
        }
    } else {   // published even after an abort (as zeros), so that the reducer does not wait in vain
        for (int i = tid; i < RD; i += kFThreads) st_tagged(a.ybuf + (size_t)slot * H + ei * RD + i, 0.f, xtag);
    }
    // ---------------------------------------------------------------- 6. combine: the shared expert's CTA per row block
    if (shared_cluster) {
        for (int o = ei * RD + tid; o < (ei + 1) * RD; o += kFThreads) {
            uint64_t v[kMaxSlots];
#pragma unroll
            for (int j = 0; j < kMaxSlots; ++j) v[j] = (j < NC) ? ld_tagged(a.ybuf + (size_t)j * H + o) : 0ull;
            const uint64_t t0 = globaltimer();
            while (true) {
                bool all = true;
#pragma unroll
                for (int j = 0; j < kMaxSlots; ++j)
                    if (j < NC && tag_of(v[j]) != xtag) {
                        all = false;
                        v[j] = ld_tagged(a.ybuf + (size_t)j * H + o);
                    }
                if (all) break;
                if (globaltimer() - t0 > kWaitLimitNs) {
                    raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT);
                    break;
                }
            }
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxSlots; ++j) s += (j < NC) ? val_of(v[j]) : 0.f;
            a.out[o] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
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
static bool codes_map(CUtensorMap* m, const uint32_t* codes, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      int bits) {
    EncodeTiledFn2 fn = encode_fn2();
    if (!fn) return false;
    const uint64_t words = cols * bits / 32;   // code words per row
    const cuuint64_t dims[2] = {words, rows};
    const cuuint64_t strides[1] = {words * 4};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int code_of(const moe_w4_layer& L) {
    return code_bits_of(L) == 4 ? kCodeU4 : (codes_e4m3(L) ? kCodeE4M3 : kCodeU8);
}

// The instance for the layer's shape and codes: specialised for the sizes of the
// pages' layer (H=2048, I=512, E=256, top-8), generic otherwise; one-byte codes
// have the specialised instance only.
using FusedKernel = void (*)(FusedArgs, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap);
static FusedKernel fused_kernel_for(const moe_w4_layer& L) {
    const bool spec = L.H == 2048 && L.I == 512 && L.E == 256 && L.top_k == 8;
    switch (code_of(L)) {
        case kCodeU4: return spec ? decode_fused_kernel<2048, 512, 256, 8, kCodeU4> : decode_fused_kernel<0, 0, 0, 0, kCodeU4>;
        case kCodeU8: return spec ? decode_fused_kernel<2048, 512, 256, 8, kCodeU8> : nullptr;
        default: return spec ? decode_fused_kernel<2048, 512, 256, 8, kCodeE4M3> : nullptr;
    }
}

static bool shape_ok(const moe_w4_layer& L) {
    const int bits = code_bits_of(L);
    if (!fused_kernel_for(L)) return false;
    if (L.H % 256 || L.I % 256 || L.H > 4096 || L.I > 2048) return false;   // slices of 16 rows; <= 16 row tiles
    if (L.H * bits / 1024 > 16) return false;                                 // gate/up box barriers
    if (L.E < 128 || L.E > 256 || L.E % 32) return false;   // top-k: 8 scores per lane; 2E floats hold the K-split partials
    if (L.top_k + 1 > kMaxSlots) return false;
    if (L.H > 64 * kPE * (L.top_k + 1)) return false;   // <= 64 router rows per CTA (32 per thread)
    const FusedSmem s(L.H, L.E, L.I, bits);
    return s.total + 1024 + 1024 <= 227 * 1024;   // + static shared memory of the kernel
}

static size_t fused_smem(const moe_w4_layer& L) { return FusedSmem(L.H, L.E, L.I, code_bits_of(L)).total + 1024; }

static cudaLaunchConfig_t fused_config(const moe_w4_layer& L, cudaLaunchAttribute* attr, cudaStream_t st,
                                       bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((L.top_k + 1) * kPE);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = fused_smem(L);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cfg;
}

// The kernel's exchanges wait on other CTAs, so every cluster must be resident
// at once: the answer of the occupancy calculator is checked (and cached per
// device and launch shape) before the fused path is taken.
bool decode_fused_supported(const moe_w4_layer& L) {
    if (!shape_ok(L)) return false;
    struct Entry { int dev, k; size_t smem; FusedKernel kern; bool ok; };
    static Entry cache[16] = {};
    static int ncache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const size_t smem = fused_smem(L);
    const FusedKernel kern = fused_kernel_for(L);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].k == L.top_k && cache[i].smem == smem && cache[i].kern == kern)
            return cache[i].ok;
    bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
              cudaSuccess;
    if (ok) {
        cudaLaunchAttribute attr[2];
        const cudaLaunchConfig_t cfg = fused_config(L, attr, nullptr, false);
        int nclusters = 0;
        ok = cudaOccupancyMaxActiveClusters(&nclusters, (void*)kern, &cfg) == cudaSuccess &&
             nclusters >= (L.top_k + 1) * kFusedClustersPerExpert;
    }
    cudaGetLastError();   // a refused query leaves no sticky error behind
    if (ncache < 16) cache[ncache++] = Entry{dev, L.top_k, smem, kern, ok};
    return ok;
}

cudaError_t launch_decode_fused(const moe_w4_layer& L, const uint16_t* x, uint16_t* out, const DecodeWs& d,
                                cudaStream_t st) {
    const int H = L.H, E = L.E, I = L.I, k = L.top_k;
    const int RG = I / kPE, RD = H / kPE, b = code_bits_of(L);
    CUtensorMap mg, mu, md, msg, msu, msd;
    bool ok = codes_map(&mg, L.gate.codes, (uint64_t)E * I, H, RG, b) &&
              codes_map(&mu, L.up.codes, (uint64_t)E * I, H, RG, b) &&
              codes_map(&md, L.down.codes, (uint64_t)E * H, I, RD, b) && codes_map(&msg, L.sh_gate.codes, I, H, RG, b) &&
              codes_map(&msu, L.sh_up.codes, I, H, RG, b) && codes_map(&msd, L.sh_down.codes, H, I, RD, b);
    if (!ok) return cudaErrorInvalidValue;
    FusedArgs a{};
    a.x = x; a.router_w = L.router_w; a.router_bias = L.router_bias; a.shared_gate = L.shared_gate;
    a.gs = L.gate.scales; a.gb = L.gate.biases; a.us = L.up.scales; a.ub = L.up.biases;
    a.ds = L.down.scales; a.db = L.down.biases;
    a.sgs = L.sh_gate.scales; a.sgb = L.sh_gate.biases; a.sus = L.sh_up.scales; a.sub = L.sh_up.biases;
    a.sds = L.sh_down.scales; a.sdb = L.sh_down.biases;
    a.cpart = d.fused_cpart; a.hx = d.fused_hx; a.ybuf = d.fused_ybuf;
    a.idx_out = d.idx; a.w_out = d.w; a.gamma_out = d.gamma; a.out = out;
    a.ctrl = d.ctrl;
    a.H = H; a.E = E; a.I = I; a.k = k;
    cudaLaunchAttribute attr[2];
    // programmatic dependent launch: the prologue may overlap the previous kernel's tail
    const cudaLaunchConfig_t cfg = fused_config(L, attr, st, true);   // shared memory opt-in set by the support check
    return cudaLaunchKernelEx(&cfg, fused_kernel_for(L), a, mg, mu, md, msg, msu, msd);
}

}  // namespace mw4
