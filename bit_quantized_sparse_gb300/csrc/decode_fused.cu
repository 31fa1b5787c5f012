// Fused batch-1 decode: the whole layer for one token in one launch.
// ("Optimizing on-device inference for Apple Silicon", sections "Optimise the
// single-row weight path" -- groups of threads cooperate on outputs while
// reading different parts of the weight matrix -- and "Reduce intermediate
// state and traffic" -- gate/up projections fused with the gated activation,
// the output projection fused with the routing scores and the shared expert.)
//
// Grid: (k+1) expert slots x 16 CTAs, one CTA per SM, launched cooperatively
// (every CTA is resident at once, which the two exchanges below rely on).
// Slot j < k is the j-th selected expert, slot k the shared expert.  CTA i
// (0..15) of a slot owns gate/up rows [i*I/16, (i+1)*I/16) of it; each of the
// 16k routed CTAs also owns output rows [c*DR, (c+1)*DR), DR = H/(16k), of the
// down projection of all k+1 slots.
//
//   1. router: routed CTA c sums 8 experts' scores x . W_r[:, e] over a
//      quarter of the H rows (these W_r loads go out first) and publishes the
//      partials; every CTA also forms the shared gate sigmoid(x . g) itself.  Every value that crosses CTAs
//      is an 8-byte (value, call tag) word, so that a reader polls the data
//      itself rather than a counter and then the data.
//   2. every routed CTA polls the E scores (bounded wait), one warp selects
//      the top-k (sorted candidate lists) and at once issues the TMA loads of
//      the CTA's gate/up slices of its slot's expert and of its down rows of
//      the k selected experts.  The shared expert needs no routing: its gate/up
//      slices, and every routed CTA's down rows of it, are requested at kernel
//      start, before the wait for the preceding kernel.
//   3. gate/up GEMV on the tensor cores as a dot-product engine: mma.sync
//      m16n8k16 with fp16 A = 1024 + q (even nibbles) or 1024 + 16 q (odd
//      nibbles), one bitwise op per pair, and B = x in fp16 with the odd
//      positions divided by 16; fp32 accumulation per 64-column group, then
//      s*(acc - 1024*sum(B)) + b*sum(x).  SwiGLU in fp32.  The instances for
//      one-byte codes take 1024 + q (8-bit codes) or the exact E4M3 value (no
//      offset) for bytes (0, 2) and (1, 3) of a word, with B in matching
//      4-column units and no division by 16.
//   4. h: every CTA publishes its slice of h as fp16 pairs already in the
//      dot engine's B-operand order; each routed CTA waits (bounded) until the
//      h of all k+1 slots carries the call's tag.
//   5. down GEMV of its DR output rows for all k+1 slots, the same dot engine,
//      each slot's rows scaled by its routing weight (the shared one by the
//      shared gate) and added in slot order in fp32; the CTA writes its rows of
//      the bf16 output.  No further exchange.
// No step waits on another CTA except these two bounded exchanges.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mw4 {

#ifndef MW4_FUSED_THREADS
#define MW4_FUSED_THREADS 512
#endif
constexpr int kPE = 16;                 // CTAs per expert slot
constexpr int kFThreads = MW4_FUSED_THREADS;   // warps hide the dot engine's latencies
constexpr int kFWarps = kFThreads / 32;
constexpr int kMaxSlots = 9;            // k + 1 <= 9
constexpr int kRE = 8;                  // router: experts per CTA (one 32-byte sector of a W_r row)
constexpr int kMaxRouterRows = 4;       // router: H rows per thread, at most
constexpr int kScoreReplicas = 8;       // copies of the published score partials (readers spread over them)
constexpr int kHReplicas = 8;           // copies of the published h and its piece sums
constexpr int kGuParts = 4;             // gate/up code slices arrive in this many parts (one barrier each)
constexpr int kDnUnits = (kMaxSlots * 8 + kFWarps - 1) / kFWarps;   // down units per warp and pass
constexpr int kDnUnitWords = 40;        // a down unit's h: 32 words (64 fp16 values), 8 piece sums

struct FusedArgs {
    const uint16_t* x;          // [H] bf16
    const float* router_w;      // [H][E]
    const float* router_bias;   // [E] or NULL
    const float* shared_gate;   // [H]
    const uint16_t* gs; const uint16_t* gb; const uint16_t* us; const uint16_t* ub;   // routed gate/up s, b
    const uint16_t* ds; const uint16_t* db;                                             // routed down s, b
    const uint16_t* sgs; const uint16_t* sgb; const uint16_t* sus; const uint16_t* sub; // shared
    const uint16_t* sds; const uint16_t* sdb;
    uint64_t* scores;           // [kScoreReplicas][RS][E] partial router scores, tagged with the call
    uint64_t* hx;               // [kHReplicas][k+1][I/2] h as fp16 pairs in B order, tagged with the call
    uint64_t* hsx;              // [kHReplicas][k+1][I/16][2] per 16 values of h: sums of the stored B values
                                // and of h itself, tagged with the call
    int32_t* idx_out;           // [k] (for inspection)
    float* w_out;               // [k]
    float* gamma_out;           // [1]
    uint16_t* out;              // [H] bf16
    Ctrl* ctrl;
    int H, E, I, k;
};

// smem carve-up (byte offsets from a 1024-aligned base), computed on both sides.
// After the gate/up GEMV its code slices are dead: each warp's copy of the h
// (in B order) and 16-value piece sums of its down units then lives in the gate
// codes region, the down partial sums and row sums in the up one.
struct FusedSmem {
    uint32_t gcodes, ucodes, dcodes, dslot, gsb, usb, dsb, xperm, xsum, xbs, logits, gred, gsum, usum, wred,
        misc, total;
    uint32_t hwarp, dred;   // aliases (see above)
    uint32_t code_region;              // bytes of one gate/up code region
    int RG, DR, NS;
    __host__ __device__ FusedSmem(int H, int E, int I, int k, int bits) {
        RG = I / kPE;
        DR = H / (kPE * k);
        NS = k + 1;
        uint32_t o = 0;
        auto take = [&](uint32_t bytes, uint32_t align) {
            o = (o + align - 1) / align * align;
            const uint32_t at = o;
            o += bytes;
            return at;
        };
        code_region = RG * H / 8 * bits;
        gcodes = take(code_region, 1024);
        ucodes = take(code_region, 1024);
        dslot = (DR * I / 8 * bits + 1023) / 1024 * 1024;   // each slot's boxes 1024-aligned (128-byte swizzle)
        dcodes = take(NS * dslot, 1024);
        gsb = take(2 * RG * (H / 64) * 2, 16);   // scales then biases
        usb = take(2 * RG * (H / 64) * 2, 16);
        dsb = take(NS * 2 * DR * (I / 64) * 2, 16);   // per slot: scales [DR][I/64] then biases
        xperm = take(H * 2, 16);
        xsum = take(H / 64 * 4, 16);
        xbs = take(H / 64 * 4, 16);
        logits = take(E * 4, 16);
        // per (row tile, warp) 16 partial row sums; before the GEMV the polled score
        // partials [RS][E] (RS * E = 128 k)
        gred = take((2 * RG * kFWarps > 128 * k ? 2 * RG * kFWarps : 128 * k) * 4, 16);
        gsum = take(RG * 4, 16);
        usum = take(RG * 4, 16);
        wred = take(kFWarps * (kRE + 1) * 4, 16);
        misc = take(512, 16);
        total = o;
        hwarp = gcodes;                 // [warp][kDnUnits * kDnUnitWords]
        dred = ucodes;                  // [NS * (I/64) * DR/16][16], then [NS][DR] row sums
    }
    // the aliased buffers fit their regions
    __host__ __device__ bool aliases_fit(int I) const {
        return (uint32_t)(kFWarps * kDnUnits * kDnUnitWords * 4) <= code_region &&
               (uint32_t)((NS * (I / 64) * DR + NS * DR) * 4) <= code_region;
    }
};

// --------------------------------------------------------------------------- legacy-MMA dot engine
MW4_DEV void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

MW4_DEV uint32_t ld_acquire_u32(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
MW4_DEV void st_relaxed_u32(unsigned int* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
// A tagged word that carries a pair of fp16 values (B-operand order) instead of a float.
MW4_DEV void st_tagged_u32(uint64_t* p, uint32_t v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | v;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(w) : "memory");
}

// Code formats of the one-kernel decode: unsigned 4-bit, unsigned 8-bit, FP8 E4M3.
enum : int { kCodeU4 = 0, kCodeU8 = 1, kCodeE4M3 = 2 };

// The B fragments of one 64-column group for this lane (8 words): 4-bit codes
// the 16-byte entries of its two 32-column blocks, one-byte codes the 8-byte
// units of its four 16-column chunks.
template <int CODE>
MW4_DEV void load_bfrag(const uint4* bperm, int grp, uint32_t (&b)[8]) {
    const int c = threadIdx.x & 3;
    if (CODE == kCodeU4) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 v = bperm[(grp * 2 + h) * 4 + c];
            b[4 * h] = v.x; b[4 * h + 1] = v.y; b[4 * h + 2] = v.z; b[4 * h + 3] = v.w;
        }
    } else {
        const uint2* bp = reinterpret_cast<const uint2*>(bperm);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint2 v = bp[(grp * 4 + h) * 4 + c];
            b[2 * h] = v.x; b[2 * h + 1] = v.y;
        }
    }
}

// The dot engine: mma.sync m16n8k16 with the weights as A (16 rows x 16
// columns) and the activation as column 0 of B; per 64-column group
// w = s*q + b, so a row's dot is s * (sum of q*value) + b * (sum of values),
// finished in fp32 by the callers.
// The A fragment of one MMA from a thread's two code words (rows r0+g and
// r0+g+8, g = lane/4), one bitwise op per register: 4-bit codes give fp16
// 1024 + q for the even nibbles of a byte and 1024 + 16 q for the odd ones
// (step 0: nibbles 0,4 and 1,5; step 1, after a shift of the word by 8:
// nibbles 2,6 and 3,7), so B holds the matching activations with the odd
// positions divided by 16 and every product is q * value + 1024 * (stored B
// value); 8-bit codes give 1024 + q for bytes (0, 2) and (1, 3); E4M3 codes
// their exact values (no offset).
// Code tiles are TMA boxes of 32 words x `rows` rows, 128-byte swizzled, box b
// at b*rows*128; a 64-column group lies inside one box.
template <int CODE>
MW4_DEV void a_frag(uint32_t wg, uint32_t wh, uint32_t (&a)[4]) {
    constexpr uint32_t M = 0x64006400u;
    if (CODE == kCodeU4) {
        a[0] = (wg & 0x000F000Fu) | M;
        a[1] = (wh & 0x000F000Fu) | M;
        a[2] = (wg & 0x00F000F0u) | M;
        a[3] = (wh & 0x00F000F0u) | M;
    } else if (CODE == kCodeE4M3) {
        e4m3x4_to_f16(wg, a[0], a[2]);
        e4m3x4_to_f16(wh, a[1], a[3]);
    } else {
        a[0] = (wg & 0x00FF00FFu) | M;
        a[1] = (wh & 0x00FF00FFu) | M;
        a[2] = ((wg >> 8) & 0x00FF00FFu) | M;
        a[3] = ((wh >> 8) & 0x00FF00FFu) | M;
    }
}

// NU independent units of one warp, each rows r0[q]..+15 of the codes tile set
// codes[q] (`rows` rows) against one 64-column group grp[q], adding to d[q] what
// group_mma adds.  The MMAs are issued step by step across the units, so that
// consecutive MMAs accumulate into different units: a unit's chain of
// dependent MMAs (24 cycles each) is covered by the other units' MMAs instead
// of stalling the warp.  B comes from shared memory per unit (bperm[q]: the
// unit's group, 8 entries of 16 bytes), or, with SHARED_B, from the registers
// `bsh` (load_bfrag) for every unit.
template <int CODE, int NU, bool SHARED_B>
MW4_DEV void units_mma(const uint8_t* const (&codes)[NU], int rows, const int (&r0)[NU], const int (&grp)[NU],
                       const uint4* const (&bperm)[NU], const uint32_t (&bsh)[8], float (&d)[NU][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    // 4-bit codes: 2 blocks of 32 columns per group, 2 MMAs per block; one-byte
    // codes: 4 chunks of 16 columns, one MMA each
    constexpr int kSteps = CODE == kCodeU4 ? 2 : 4;
    constexpr int kPerBox = CODE == kCodeU4 ? 2 : 4;   // blocks (chunks) per group
#pragma unroll
    for (int h = 0; h < kSteps; ++h) {
        uint32_t wg[NU], wh[NU], b[NU][4];
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            const int bk = grp[q] * kPerBox + h;   // block (chunk) of the group
            const uint8_t* row0 = codes[q] + (size_t)(bk >> 3) * rows * 128 + (r0[q] + g) * 128 + c * 4 +
                                  (((bk & 7) ^ g) << 4);
            wg[q] = *reinterpret_cast<const uint32_t*>(row0);
            wh[q] = *reinterpret_cast<const uint32_t*>(row0 + 8 * 128);
            if (SHARED_B) {
                if (CODE == kCodeU4) {
                    b[q][0] = bsh[4 * h]; b[q][1] = bsh[4 * h + 1]; b[q][2] = bsh[4 * h + 2]; b[q][3] = bsh[4 * h + 3];
                } else {
                    b[q][0] = bsh[2 * h]; b[q][1] = bsh[2 * h + 1];
                }
            } else if (CODE == kCodeU4) {
                const uint4 v = bperm[q][h * 4 + c];
                b[q][0] = v.x; b[q][1] = v.y; b[q][2] = v.z; b[q][3] = v.w;
            } else {
                const uint2 v = reinterpret_cast<const uint2*>(bperm[q])[h * 4 + c];
                b[q][0] = v.x; b[q][1] = v.y;
            }
        }
#pragma unroll
        for (int q = 0; q < NU; ++q) {
            uint32_t a[4];
            a_frag<CODE>(wg[q], wh[q], a);
            mma_f16_16816(d[q], a, b[q][0], b[q][1]);
        }
        if (CODE == kCodeU4) {
#pragma unroll
            for (int q = 0; q < NU; ++q) {
                uint32_t a[4];
                a_frag<CODE>(wg[q] >> 8, wh[q] >> 8, a);
                mma_f16_16816(d[q], a, b[q][2], b[q][3]);
            }
        }
    }
}

// The four B-operand words of 8 consecutive activation values v[0..7] (an
// entry of 16 bytes): 4-bit codes (v0, v4), (v1, v5)/16, (v2, v6), (v3, v7)/16;
// one-byte codes the 4-column units (v0, v2), (v1, v3), (v4, v6), (v5, v7).
template <int CODE>
MW4_DEV uint32_t b_word(const float (&v)[8], int m) {
    if (CODE == kCodeU4) {
        const int a = m >> 1 ? 2 : 0, o = m & 1;   // m: 0 -> (0,4), 1 -> (1,5)/16, 2 -> (2,6), 3 -> (3,7)/16
        const float sc = o ? 0.0625f : 1.0f;
        return h2_as_u32(__floats2half2_rn(v[a + o] * sc, v[a + o + 4] * sc));
    }
    const int b = (m >> 1) * 4 + (m & 1);   // m: 0 -> (0,2), 1 -> (1,3), 2 -> (4,6), 3 -> (5,7)
    return h2_as_u32(__floats2half2_rn(v[b], v[b + 2]));
}

// Group sums of one 16-byte B entry as stored: `sb` of the pairs that carry
// the 1024 offset unscaled, `so` of the pairs divided by 16 (4-bit codes).
template <int CODE>
MW4_DEV void b_entry_sums(const uint4& q, float& sb, float& so) {
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(u32_as_h2(u[j]));
        if (CODE == kCodeU4 && (j & 1)) so += f.x + f.y; else sb += f.x + f.y;
    }
}

// 3-D tiled load: code rows seen as [box column][row][32 words], so that one copy
// brings several 128-byte box columns of a row slice (each landing as a 2-D box
// of `rows` x 128 bytes, one after the other); c2 is the first box column.
MW4_DEV void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Bounded wait on an mbarrier phase that ignores the abort flag: used before
// exit so that no TMA copy of this CTA is still in flight when it leaves.
static __device__ __noinline__ void mbar_drain(uint64_t* bar) {
    if (mbar_try_wait(bar, 0)) return;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, 0))
        if (globaltimer() - t0 > kWaitLimitNs) return;
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
    const FusedSmem L(H, E, I, k, kBits);
    const int RG = L.RG, DR = L.DR, NS = L.NS;
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
    float* logits = reinterpret_cast<float*>(sm + L.logits);
    float* gred = reinterpret_cast<float*>(sm + L.gred);
    float* gsum = reinterpret_cast<float*>(sm + L.gsum);
    float* usum = reinterpret_cast<float*>(sm + L.usum);
    float* wred = reinterpret_cast<float*>(sm + L.wred);
    uint32_t* hwarp = reinterpret_cast<uint32_t*>(sm + L.hwarp);   // after the gate/up GEMV
    float* dred = reinterpret_cast<float*>(sm + L.dred);
    uint8_t* misc = sm + L.misc;
    // TMA boxes of 128-byte code rows: 256 columns of 4-bit codes, 128 of one-byte codes.
    // Gate/up slices come in kGuParts parts of their box columns (one 3-D copy per
    // matrix and part, one barrier per part, so the GEMV starts on the first part),
    // each slot's down rows in one 3-D copy.
    const int nbox_gu = H * kBits / 1024;
    uint64_t* bar_gu = reinterpret_cast<uint64_t*>(misc);               // [kGuParts] parts of the gate/up slices
    uint64_t* bar_dn = bar_gu + kGuParts;                                // routed down rows
    uint64_t* bar_dsh = bar_dn + 1;                                      // shared expert's down rows
    uint64_t* bar_sb = bar_dsh + 1;                                      // gate/up scales, biases (warp 0's cp.async)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_sb + 1);
    int* sel_e = reinterpret_cast<int*>(bar_sb + 2);                     // [kMaxSlots] selected experts
    float* sel_w = reinterpret_cast<float*>(sel_e + kMaxSlots);          // [kMaxSlots] weights (slot k: gamma)
    uint32_t* xtag_s = reinterpret_cast<uint32_t*>(sel_w + kMaxSlots);   // this call's exchange tag
    uint32_t* xinj_s = xtag_s + 1;                                       // test hook: skip a publish
    int* issued = reinterpret_cast<int*>(xtag_s + 2);   // bits: 0 gate/up codes, 1 down, 2 shared down, 3 gate/up s, b

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = blockIdx.x, slot = G / kPE, ei = G % kPE;
    const int NR = k * kPE;                       // routed CTAs (also the down CTAs)
    const bool shared_cta = (slot == k);
    const bool down_cta = G < NR;
    unsigned int* status = &a.ctrl->status;
    // Router: with EG = E/8 groups of 8 experts and RS = NR/EG splits of the H rows,
    // CTA G < EG*RS sums experts [eg*8, eg*8+8) over rows [rs*H/RS, (rs+1)*H/RS)
    // (eg = G % EG, rs = G / EG): one full 32-byte sector per W_r row it reads.
    const int EG = E / kRE, RS = NR / EG, r_rows = H / RS;
    const bool router_cta = G < EG * RS;
    const int r_eg = G % EG, r_rs = G / EG;
    constexpr int kRPT = (kH && kE && kK) ? (kH / ((kK * kPE) / (kE / kRE)) + kFThreads - 1) / kFThreads
                                          : kMaxRouterRows;   // router rows per thread
    constexpr int kGPT = kH ? (kH + kFThreads - 1) / kFThreads : 8;   // shared-gate rows per thread
    const int gdrow_sh = G * DR;                  // this CTA's down rows (routed CTAs)
    const int dchunks = DR * (I / 64) * 2 / 16;   // 16-byte pieces of one slot's down scales (or biases)

    // The barriers first: their initialisation is published with a release fence,
    // which must not wait for the router loads below.
    if (tid == 0) {
        for (int q = 0; q < kGuParts; ++q) mbar_init(&bar_gu[q], 1);
        mbar_init(bar_dn, 1);
        mbar_init(bar_dsh, 1);
        mbar_init(bar_sb, 1);
        *abort_flag = 0;
        *issued = 0;
        fence_mbar_init();
    }
    // The kernel may start before the previous kernel on the stream has finished
    // (programmatic dependent launch): until griddep_wait() it touches only
    // weights, its own shared memory and the tensor maps.
    // Router weights first: thread t holds row r_rs*H/RS + t (+ kFThreads, ...) of W_r
    // for the CTA's 8 experts, and the shared gate at rows t, t + kFThreads, ...
    // The loads are unconditional (row indices clamped into range, the surplus
    // rows' x taken as 0 later), so that nothing before griddep_wait() waits on them.
    float rw[kRPT][kRE], rg[kGPT];
    if (router_cta) {
#pragma unroll
        for (int i = 0; i < kRPT; ++i) {
            const int h = min(r_rs * r_rows + min(tid + i * kFThreads, r_rows - 1), H - 1);
            const float4* src = reinterpret_cast<const float4*>(a.router_w + (size_t)h * E + r_eg * kRE);
            const float4 w0 = __ldg(src), w1 = __ldg(src + 1);
            rw[i][0] = w0.x; rw[i][1] = w0.y; rw[i][2] = w0.z; rw[i][3] = w0.w;
            rw[i][4] = w1.x; rw[i][5] = w1.y; rw[i][6] = w1.z; rw[i][7] = w1.w;
        }
    }
    float rbias[8];   // warp 0 of a routed CTA: the router bias of experts lane + 32 i
    if (down_cta) {
#pragma unroll
        for (int i = 0; i < kGPT; ++i) rg[i] = __ldg(a.shared_gate + min(tid + i * kFThreads, H - 1));
        if (warp == 0 && a.router_bias) {
#pragma unroll
            for (int i = 0; i < 8; ++i) rbias[i] = __ldg(a.router_bias + min(lane + 32 * i, E - 1));
        }
    }
    if (tid == 32) {   // the descriptors are fetched once, early, off the critical path
        prefetch_tensormap(&mg); prefetch_tensormap(&mu); prefetch_tensormap(&md);
        prefetch_tensormap(&msg); prefetch_tensormap(&msu); prefetch_tensormap(&msd);
    }
    __syncthreads();

    // ---------------------------------------------------------------- weight loads
    // gate/up code slices of expert e (E = the shared expert), by one thread: two
    // halves of the box columns, each half of gate and of up on one barrier
    auto issue_gateup = [&](int e) {
        const bool sh = (e >= E);
        const int grow = (sh ? 0 : e * I) + ei * RG;
        const int hb = nbox_gu / kGuParts;   // box columns per part
        const uint32_t gsz = RG * (H / 64) * 2;   // one scale (or bias) slice
        const size_t go = (size_t)grow * (H / 64);
        mbar_arrive_expect_tx(bar_sb, 4 * gsz);
        bulk_load(gsb, (sh ? a.sgs : a.gs) + go, gsz, bar_sb);
        bulk_load(gsb + RG * (H / 64), (sh ? a.sgb : a.gb) + go, gsz, bar_sb);
        bulk_load(usb, (sh ? a.sus : a.us) + go, gsz, bar_sb);
        bulk_load(usb + RG * (H / 64), (sh ? a.sub : a.ub) + go, gsz, bar_sb);
        for (int h = 0; h < kGuParts; ++h) {
            mbar_arrive_expect_tx(&bar_gu[h], 2u * hb * RG * 128);
            tma_load_3d(gcodes + (size_t)h * hb * RG * 128, sh ? &msg : &mg, 0, grow, h * hb, &bar_gu[h]);
            tma_load_3d(ucodes + (size_t)h * hb * RG * 128, sh ? &msu : &mu, 0, grow, h * hb, &bar_gu[h]);
        }
    };
    // down code rows [G*DR, (G+1)*DR) of expert e into slot j's region, by one thread
    auto issue_down = [&](int j, int e, uint64_t* bar) {
        const int drow = (e >= E ? 0 : e * H) + gdrow_sh;
        tma_load_3d(dcodes + (size_t)j * L.dslot, e >= E ? &msd : &md, 0, drow, 0, bar);
    };
    // the down rows' scales and biases by cp.async, one 16-byte piece per call:
    // piece c of slot j's down rows of expert e (2 dchunks: s, b)
    auto sb_down = [&](int j, int e, int c) {
        const bool sh = (e >= E);
        const size_t dO = (size_t)((sh ? 0 : e * H) + gdrow_sh) * (I / 64);
        const int arr = c / dchunks, o = (c % dchunks) * 8;
        const uint16_t* src = arr == 0 ? (sh ? a.sds : a.ds) : (sh ? a.sdb : a.db);
        cp_async_16(dsb + (size_t)j * 2 * DR * (I / 64) + arr * DR * (I / 64) + o, src + dO + o);
    };
    const uint32_t dn_bytes = (uint32_t)DR * (I * kBits / 8);   // one slot's down code rows
    if (shared_cta) {   // the shared expert needs no routing: its loads go out now
        if (tid == 0) {
            issue_gateup(E);
            *issued |= 1 | 8;
        }
    } else {            // routed CTAs: their down rows of the shared expert
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_dsh, dn_bytes);
            issue_down(k, E, bar_dsh);
            *issued |= 4;
        }
        for (int c = tid; c < 2 * dchunks; c += kFThreads) sb_down(k, E, c);
    }
    cp_async_commit();

    griddep_wait();   // from here on: x, the workspace and its counters
    // Values crossing CTAs carry this call's tag (the call counter + 1, never 0):
    // a reader polls the data itself.  The counter advances once a routed CTA has
    // seen every slot's h with the tag (so every CTA has read the counter), or
    // when a CTA gives up.
    if (tid == 0) {
        uint32_t t = ld_acquire_u32(&a.ctrl->pad[kCtrlEpochWord]) + 1u;
        *xtag_s = t ? t : 1u;
        *xinj_s = ld_acquire_u32(&a.ctrl->pad[kCtrlInjectWord]);
    }

    // ---------------------------------------------------------------- 1. router partial scores and the shared gate
    if (down_cta) {
        float acc[kRE + 1];
#pragma unroll
        for (int c = 0; c <= kRE; ++c) acc[c] = 0.f;
        if (router_cta) {
#pragma unroll
            for (int i = 0; i < kRPT; ++i) {
                const int hr = tid + i * kFThreads;
                const float xv = hr < r_rows ? bf16_bits_to_float(__ldg(a.x + r_rs * r_rows + hr)) : 0.f;
#pragma unroll
                for (int c = 0; c < kRE; ++c) acc[c] = fmaf(xv, rw[i][c], acc[c]);
            }
        }
#pragma unroll
        for (int i = 0; i < kGPT; ++i) {
            const int h = tid + i * kFThreads;
            const float xv = h < H ? bf16_bits_to_float(__ldg(a.x + h)) : 0.f;
            acc[kRE] = fmaf(xv, rg[i], acc[kRE]);
        }
#pragma unroll
        for (int c = 0; c <= kRE; ++c) {
            const float v = warp_sum(acc[c]);
            if (lane == 0) wred[warp * (kRE + 1) + c] = v;
        }
    }
    __syncthreads();
    const uint32_t xtag = *xtag_s;
    if (down_cta && tid <= kRE * kScoreReplicas) {
        // block sums in warp order: the 8 partial scores, each published to every
        // replica (thread c + 8 r: expert c, replica r), and the shared gate
        const int c = tid < kRE * kScoreReplicas ? tid % kRE : kRE;
        float sum = 0.f;
        for (int w = 0; w < kFWarps; ++w) sum += wred[w * (kRE + 1) + c];
        if (c == kRE) {
            sel_w[k] = 1.0f / (1.0f + expf(-sum));
            if (G == 0) *a.gamma_out = sel_w[k];
        } else if (router_cta && !(*xinj_s != 0u && G == 0)) {
            const int r = tid / kRE;
            st_tagged(a.scores + ((size_t)r * RS + r_rs) * E + r_eg * kRE + c, sum, xtag);
        }
    }

    // ---------------------------------------------------------------- 2. scores in, top-k, loads (routed CTAs)
    // warps 0 .. RS-1 each poll one row split's partials of all E experts in this
    // CTA's replica (bounded wait) and leave them in shared memory; warp 0 then adds
    // them in split order, selects the top-k and issues the loads
    if (!shared_cta && warp < RS) {
        constexpr int kNV = 8;   // E <= 256 scores: lane l holds experts l + 32 i
        const uint64_t* src = a.scores + ((size_t)(G % kScoreReplicas) * RS + warp) * E;
        uint64_t v[kNV];
#pragma unroll
        for (int i = 0; i < kNV; ++i) v[i] = (lane + 32 * i < E) ? ld_tagged(src + lane + 32 * i) : 0ull;
        const uint64_t t0 = globaltimer();
        bool ok = true;
        for (int it = 1;; ++it) {
            bool all = true;
#pragma unroll
            for (int i = 0; i < kNV; ++i)
                if (lane + 32 * i < E && tag_of(v[i]) != xtag) {
                    all = false;
                    v[i] = ld_tagged(src + lane + 32 * i);
                }
            if (__all_sync(0xffffffffu, all)) break;
            if ((it & 15) == 0 && globaltimer() - t0 > kWaitLimitNs) { ok = false; break; }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) { raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT); *abort_flag = 1; }
        } else {
            float* part = gred + warp * E;   // gred is free until the gate/up GEMV
#pragma unroll
            for (int i = 0; i < kNV; ++i)
                if (lane + 32 * i < E) part[lane + 32 * i] = val_of(v[i]);
        }
        asm volatile("bar.sync 1, %0;" :: "r"(RS * 32) : "memory");   // the polling warps only
    }
    int rsel = -1;      // warp 0 of a routed CTA: lane j < k holds the j-th selection
    float rval = 0.f;   // and its score
    if (!shared_cta && warp == 0) {
        if (!*abort_flag) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                if (e < E) {
                    float sum = 0.f;
                    for (int r = 0; r < RS; ++r) sum += gred[r * E + e];
                    logits[e] = sum + (a.router_bias ? rbias[i] : 0.f);
                }
            }
            __syncwarp();
            int sidx;
            float sval;
            warp_topk_sorted<8>(logits, E, k, sidx, sval);
            const bool bad = __any_sync(0xffffffffu, lane < k && (sidx < 0 || sidx >= E));
            if (bad) {
                if (lane == 0) { raise_status(status, MOE_W4_STATUS_BAD_INDEX); *abort_flag = 1; }
            } else {
                // what the gate/up GEMV needs first: its code slices and their scales
                // and biases; the down rows and the routing weights follow once the
                // block has the selection
                const int e_mine = __shfl_sync(0xffffffffu, sidx, slot);
                if (lane == 0) {
                    issue_gateup(e_mine);
                    *issued |= 1 | 8;
                }
                if (lane < k) sel_e[lane] = sidx;
                rsel = sidx;
                rval = sval;
            }
        }
    }
    if (shared_cta || warp >= RS) {
        // x as fp16 B fragments, one thread per 16-byte entry (entry i holds the B
        // words of x[8i .. 8i+7], b_word), plus the per-64-column group sums of the
        // stored values (xbs) and of the values the products use (xsum), reduced
        // over the 8 lanes of a group.  Routed CTAs: the warps that do not poll the
        // scores (H/8 is a multiple of 32, so every warp runs whole iterations).
        const int t0 = shared_cta ? tid : tid - 32 * RS, nt = shared_cta ? kFThreads : kFThreads - 32 * RS;
        for (int i = t0; i < H / 8; i += nt) {
            const uint4 q = *reinterpret_cast<const uint4*>(a.x + i * 8);
            const uint32_t e[4] = {q.x, q.y, q.z, q.w};   // pairs (0,1) (2,3) (4,5) (6,7)
            float f[8];
            bool bad = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = __uint_as_float(e[j] << 16);
                f[2 * j + 1] = __uint_as_float(e[j] & 0xFFFF0000u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) bad |= !(fabsf(f[j]) <= 65504.f);
            const uint4 o = make_uint4(b_word<CODE>(f, 0), b_word<CODE>(f, 1), b_word<CODE>(f, 2), b_word<CODE>(f, 3));
            reinterpret_cast<uint4*>(xperm)[i] = o;
            float sb = 0.f, so = 0.f;
            b_entry_sums<CODE>(o, sb, so);
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
    }
    __syncthreads();
    const bool run = !*abort_flag;
    if (!shared_cta && run) {
        if (warp == 0) {   // the selected experts' down rows, then the routing weights
            if (lane == 0) {
                mbar_arrive_expect_tx(bar_dn, (uint32_t)k * dn_bytes);
                *issued |= 2;
            }
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const int e = __shfl_sync(0xffffffffu, rsel, j);
                if (lane == 0) issue_down(j, e, bar_dn);
            }
            const float v0 = __shfl_sync(0xffffffffu, rval, 0);   // the largest selected score
            const float ex = lane < k ? expf(rval - v0) : 0.f;
            const float z = warp_sum(ex);
            const float w = ex / z;   // softmax over the selection
            if (lane < k) sel_w[lane] = w;
            if (G == 0 && lane < k) { a.idx_out[lane] = rsel; a.w_out[lane] = w; }
        } else {           // the other warps: the down rows' scales and biases
            const int ndn = k * 2 * dchunks;
#pragma unroll 1
            for (int c = tid - 32; c < ndn; c += kFThreads - 32)
                sb_down(c / (2 * dchunks), sel_e[c / (2 * dchunks)], c % (2 * dchunks));
        }
    }
    cp_async_commit();
    griddep_launch_dependents();   // the next kernel on the stream may start its prologue

    // ---------------------------------------------------------------- 3. gate/up GEMV
    // 2*RG/16 row tiles (gate, then up) x KS splits of the 64-column groups
    // box 0 also carries the scales/biases; the block agrees on the outcome of the wait
    const bool gu_ok = __syncthreads_and(run ? mbar_wait(bar_sb, 0, abort_flag, status) : 0);
    if (gu_ok) {
        // 2*RG/16 row tiles (gate, then up), every warp on all of them for its own
        // groups gg = warp, warp + kFWarps, ...: each group's B fragments are loaded
        // once for all the tiles, whose MMA chains are independent (fewer groups per
        // warp measured faster than spreading every part of the columns over all
        // warps: the per-group work around the MMAs is paid once per group)
        const int ntile = 2 * (RG / 16), ngrp = H / 64;
        constexpr int kTC = 4;   // row tiles per pass
        for (int t0 = 0; t0 < ntile; t0 += kTC) {
            float acc[kTC][2];
#pragma unroll
            for (int t = 0; t < kTC; ++t) acc[t][0] = acc[t][1] = 0.f;
            for (int gg = warp; gg < ngrp; gg += kFWarps) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bar_gu[gg / (ngrp / kGuParts)], 0, abort_flag, status)))
                    break;   // warp-uniform: the MMAs need the whole warp
                uint32_t bf[8];
                load_bfrag<CODE>(reinterpret_cast<const uint4*>(xperm), gg, bf);
                float d[kTC][4];
                const uint8_t* tcodes[kTC];
                int tr0[kTC], tgrp[kTC];
                const uint4* tnob[kTC];
#pragma unroll
                for (int t = 0; t < kTC; ++t) {   // a tile past the end repeats the last one, unused
                    d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
                    const int tt = min(t0 + t, ntile - 1);
                    const bool up = tt >= ntile / 2;
                    tcodes[t] = up ? ucodes : gcodes;
                    tr0[t] = (up ? tt - ntile / 2 : tt) * 16;
                    tgrp[t] = gg;
                    tnob[t] = nullptr;
                }
                units_mma<CODE, kTC, true>(tcodes, RG, tr0, tgrp, tnob, bf, d);
                const float bs = xbs[gg], xs = xsum[gg];
                const int g = lane >> 2, ngr = H / 64;
#pragma unroll
                for (int t = 0; t < kTC; ++t) {
                    const int tt = t0 + t;
                    if (tt >= ntile) break;
                    const bool up = tt >= ntile / 2;
                    const int r0 = (up ? tt - ntile / 2 : tt) * 16 + g;
                    const uint16_t* sc = up ? usb : gsb;
                    const uint16_t* bi = sc + RG * ngr;
                    acc[t][0] = fmaf(bf16_bits_to_float(sc[r0 * ngr + gg]), d[t][0] - 1024.f * bs,
                                     fmaf(bf16_bits_to_float(bi[r0 * ngr + gg]), xs, acc[t][0]));
                    acc[t][1] = fmaf(bf16_bits_to_float(sc[(r0 + 8) * ngr + gg]), d[t][2] - 1024.f * bs,
                                     fmaf(bf16_bits_to_float(bi[(r0 + 8) * ngr + gg]), xs, acc[t][1]));
                }
            }
            if ((lane & 3) == 0) {
#pragma unroll
                for (int t = 0; t < kTC; ++t)
                    if (t0 + t < ntile) {
                        gred[((t0 + t) * kFWarps + warp) * 16 + (lane >> 2)] = acc[t][0];
                        gred[((t0 + t) * kFWarps + warp) * 16 + (lane >> 2) + 8] = acc[t][1];
                    }
            }
        }
        __syncthreads();
        for (int i = tid; i < 2 * RG; i += kFThreads) {   // sum the warps' group partials in warp order
            const int t = i / 16, r = i % 16;
            float v = 0.f;
            for (int w = 0; w < kFWarps; ++w) v += gred[(t * kFWarps + w) * 16 + r];
            (t < ntile / 2 ? gsum : usum)[(t % (ntile / 2)) * 16 + r] = v;
        }
    }
    cp_async_wait<0>();   // this thread's pieces of the down scales and biases (read after the barrier)
    __syncthreads();
    // ---------------------------------------------------------------- 4. h exchange
    // this CTA's RG values of h as RG/2 tagged fp16 pairs in B order (entry q of the
    // slice = h[8q .. 8q+7]), and per 16 values of h (8 words) the sums of the
    // stored B values (with the 1024 offset) and of the values the products use;
    // published even after an abort (as zeros), so that no routed CTA waits in vain
    const bool gu_done = gu_ok && !*abort_flag;
    {   // thread t < kHReplicas * RG/2: word t % (RG/2) of the slice, to replica t / (RG/2)
        const int nwc = RG / 2;   // a multiple of 8, so whole warps and whole 8-word pieces
        if (tid < kHReplicas * nwc) {
            const int r = tid / nwc, wi = tid % nwc, q = wi >> 2, m = wi & 3;
            // word m of entry q holds two of h[8q .. 8q+7] (b_word's pairs)
            const int j0 = CODE == kCodeU4 ? m : (m >> 1) * 4 + (m & 1);
            const int j1 = j0 + (CODE == kCodeU4 ? 4 : 2);
            const float sc = (CODE == kCodeU4 && (m & 1)) ? 0.0625f : 1.0f;
            const float h0 = gu_done ? silu_f(gsum[q * 8 + j0]) * usum[q * 8 + j0] : 0.f;
            const float h1 = gu_done ? silu_f(gsum[q * 8 + j1]) * usum[q * 8 + j1] : 0.f;
            if (r == 0 && !(fabsf(h0) <= 65504.f && fabsf(h1) <= 65504.f)) raise_status(status, MOE_W4_STATUS_FP16_RANGE);
            const uint32_t wd = h2_as_u32(__floats2half2_rn(h0 * sc, h1 * sc));
            const float2 f = __half22float2(u32_as_h2(wd));
            float sb = (CODE == kCodeU4 && (m & 1)) ? 0.f : f.x + f.y;   // stored pairs at full scale
            float so = (CODE == kCodeU4 && (m & 1)) ? f.x + f.y : 0.f;   // stored pairs divided by 16
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {   // the 8 words of one 16-value piece
                sb += __shfl_xor_sync(0xffffffffu, sb, off);
                so += __shfl_xor_sync(0xffffffffu, so, off);
            }
            const size_t nw = (size_t)NS * (I / 2), ns2 = (size_t)NS * (I / 16) * 2;
            st_tagged_u32(a.hx + r * nw + (size_t)slot * (I / 2) + ei * nwc + wi, wd, xtag);
            if ((wi & 7) == 0) {
                uint64_t* hs = a.hsx + r * ns2 + ((size_t)slot * (I / 16) + ei * (RG / 16) + wi / 8) * 2;
                st_tagged(hs, CODE == kCodeE4M3 ? 0.f : sb + so, xtag);   // E4M3 products carry no 1024 offset
                st_tagged(hs + 1, sb + 16.f * so, xtag);
            }
        }
    }
    // ---------------------------------------------------------------- 5. h in, down GEMV, weighted sum, output rows
    // Units (slot, row tile, group) in slot-major order; warp w takes the contiguous
    // units [w*nunit/16, (w+1)*nunit/16), so most warps need one slot's h.  Each warp
    // polls only the h words and piece sums of its own units (bounded wait) and
    // starts its MMAs as soon as they carry the call's tag: the down products of the
    // slots that publish early overlap the wait for the late ones.  Each unit's 16
    // row sums go to dred[unit][16].
    const int ngrp = I / 64, ntl = DR / 16, nunit = NS * ntl * ngrp;
    constexpr int kU = kDnUnits;                                  // units per pass (I = 512: every unit of the warp)
    constexpr int kUW = kDnUnitWords;
    constexpr int kPW = (kU * kUW + 31) / 32;                     // polled words per lane and pass
    // (every branch below is warp-uniform: the MMAs need the whole warp)
    if (__all_sync(0xffffffffu, down_cta && gu_done && !*abort_flag)) {
        const int ua = warp * nunit / kFWarps, ub = (warp + 1) * nunit / kFWarps;
        const bool w_ok = __all_sync(0xffffffffu, mbar_wait(bar_dn, 0, abort_flag, status) &&
                                                      mbar_wait(bar_dsh, 0, abort_flag, status));
        const uint64_t* hxr = a.hx + (size_t)(G % kHReplicas) * NS * (I / 2);      // this CTA's replica
        const uint64_t* hsr = a.hsx + (size_t)(G % kHReplicas) * NS * (I / 16) * 2;
        uint32_t* wh = hwarp + warp * (kU * kUW);                                  // this warp's h and sums
        for (int u0 = ua; w_ok && u0 < ub; u0 += kU) {
            const int nu = min(kU, ub - u0), nwords = nu * kUW;
            // word i of the pass: unit u0 + i / kUW, its h word (i % kUW < 32) or piece sum
            auto src = [&](int i) {
                const int u = u0 + i / kUW, k2 = i % kUW, j = u / (ntl * ngrp), gg = u % ngrp;
                return k2 < 32 ? hxr + (size_t)j * (I / 2) + gg * 32 + k2
                               : hsr + ((size_t)j * (I / 16) + gg * 4) * 2 + (k2 - 32);
            };
            uint64_t w[kPW];
#pragma unroll
            for (int m = 0; m < kPW; ++m) {
                const int i = lane + 32 * m;
                w[m] = i < nwords ? ld_tagged(src(i)) : 0ull;
            }
            const uint64_t t0 = globaltimer();
            for (int it = 1;; ++it) {
                bool all = true;
#pragma unroll
                for (int m = 0; m < kPW; ++m) {
                    const int i = lane + 32 * m;
                    if (i < nwords && tag_of(w[m]) != xtag) {
                        all = false;
                        w[m] = ld_tagged(src(i));
                    }
                }
                if (all) break;
                if ((it & 15) == 0 && globaltimer() - t0 > kWaitLimitNs) {
                    raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
#pragma unroll
            for (int m = 0; m < kPW; ++m) {
                const int i = lane + 32 * m;
                if (i < nwords) wh[i] = (uint32_t)w[m];   // h pairs, or the float bits of a piece sum
            }
            __syncwarp();
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            // branch-free: a unit past the warp's range repeats its last one, unstored
            float d[kU][4];
            int uj[kU], ugg[kU], utl[kU];
            const uint8_t* ucodes_q[kU];
            const uint4* ub4[kU];
            const uint32_t nob[8] = {};
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int qq = min(q, nu - 1), u = u0 + qq;
                uj[q] = u / (ntl * ngrp);
                utl[q] = (u / ngrp) % ntl * 16;
                ugg[q] = u % ngrp;
                d[q][0] = d[q][1] = d[q][2] = d[q][3] = 0.f;
                ucodes_q[q] = dcodes + (size_t)uj[q] * L.dslot;
                ub4[q] = reinterpret_cast<const uint4*>(wh + qq * kUW);
            }
            units_mma<CODE, kU, false>(ucodes_q, DR, utl, ugg, ub4, nob, d);
            const int g = lane >> 2;
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int j = uj[q], gg = ugg[q], r0 = utl[q] + g;
                const uint16_t* sc = dsb + (size_t)j * 2 * DR * ngrp;
                const uint16_t* bi = sc + DR * ngrp;
                // per-64-value group sums of h: its four 16-value pieces in order
                const float* pc = reinterpret_cast<const float*>(wh + min(q, nu - 1) * kUW + 32);
                const float bs = ((pc[0] + pc[2]) + pc[4]) + pc[6], hs = ((pc[1] + pc[3]) + pc[5]) + pc[7];
                const float v0 = fmaf(bf16_bits_to_float(sc[r0 * ngrp + gg]), d[q][0] - 1024.f * bs,
                                      bf16_bits_to_float(bi[r0 * ngrp + gg]) * hs);
                const float v1 = fmaf(bf16_bits_to_float(sc[(r0 + 8) * ngrp + gg]), d[q][2] - 1024.f * bs,
                                      bf16_bits_to_float(bi[(r0 + 8) * ngrp + gg]) * hs);
                const int u = u0 + q;
                if ((lane & 3) == 0 && q < nu) {
                    dred[u * 16 + g] = v0;
                    dred[u * 16 + g + 8] = v1;
                }
            }
            __syncwarp();   // this pass's h is read before the next pass overwrites it
        }
    }
    __syncthreads();
    const bool dn_ok = down_cta && gu_done && !*abort_flag;
    // every slot's h carried the tag for one of this CTA's warps, so every CTA has read
    // the call counter
    if (dn_ok && G == 0 && tid == 0) st_relaxed_u32(&a.ctrl->pad[kCtrlEpochWord], xtag);
    if (dn_ok) {
        // out row r = sum over slots (in order) of the slot's weight times its row sum
        // over the groups (in order): the row sums y[j][r] by one thread each, then
        // the weighted sums
        float* ysl = dred + nunit * 16;   // [NS][DR]
        for (int i = tid; i < NS * DR; i += kFThreads) {
            const int j = i / DR, r = i % DR, tl = r / 16, rr = r % 16;
            float y = 0.f;
            for (int gg = 0; gg < ngrp; ++gg) y += dred[((j * ntl + tl) * ngrp + gg) * 16 + rr];
            ysl[i] = y;
        }
        __syncthreads();
        for (int r = tid; r < DR; r += kFThreads) {
            float acc = 0.f;
            for (int j = 0; j < NS; ++j) acc = fmaf(sel_w[j], ysl[j * DR + r], acc);
            a.out[gdrow_sh + r] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        }
    }
    // ---------------------------------------------------------------- exit
    // a CTA that gave up advances the call counter itself (the tags of this call's
    // words must not be taken for the next call's), and no TMA copy of this CTA
    // may still be in flight when it leaves (without an abort every barrier has
    // already been waited on)
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        st_relaxed_u32(&a.ctrl->pad[kCtrlEpochWord], xtag);
        const int is = *issued;
        if (is & 1) {
            for (int q = 0; q < kGuParts; ++q) mbar_drain(&bar_gu[q]);
        }
        if (is & 2) mbar_drain(bar_dn);
        if (is & 4) mbar_drain(bar_dsh);
        if (is & 8) mbar_drain(bar_sb);
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
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn2>(p);
    });
    return fn;
}

// codes [rows][cols/8] uint32 seen as [cols/256 box columns][rows][32 words]
// (dimension 1 = rows, dimension 2 = box columns 128 bytes apart), box = 32
// words x box_rows x box_cols; every (row, box column) lands as one 128-byte
// line, 128-byte swizzled, box column c of the copy at c*box_rows*128.
static bool codes_map(CUtensorMap* m, const uint32_t* codes, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t box_cols, int bits) {
    EncodeTiledFn2 fn = encode_fn2();
    if (!fn) return false;
    const uint64_t words = cols * bits / 32;   // code words per row
    const cuuint64_t dims[3] = {32, rows, words / 32};
    const cuuint64_t strides[2] = {words * 4, 128};
    const cuuint32_t box[3] = {32, box_rows, box_cols};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(codes), dims, strides, box, estr,
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
    const int bits = code_bits_of(L), k = L.top_k;
    if (!fused_kernel_for(L)) return false;
    if (k < 1 || k + 1 > kMaxSlots) return false;
    if (L.H % 256 || L.I % 256 || L.H > 4096 || L.I > 2048) return false;   // slices of 16 rows; <= 16 row tiles
    if (L.H % (kPE * k * 16)) return false;                                   // down rows per CTA: whole m16 tiles
    if (L.H * bits / 1024 > 16 || (L.H * bits / 1024) % kGuParts) return false;   // gate/up: parts of box columns
    if (L.E < 128 || L.E > 256 || L.E % 32) return false;                     // top-k: 8 scores per lane
    const int EG = L.E / kRE, NR = k * kPE;                                   // router: 8 experts per CTA
    if (EG > NR || NR % EG || NR / EG > 8 || L.H % (NR / EG)) return false;   // row splits: at most 8 polling warps
    if (L.H / (NR / EG) > kMaxRouterRows * kFThreads || L.H > 8 * kFThreads) return false;
    if (L.I / 64 * (k + 1) > 9 * 8) return false;                             // down units per warp in flight
    if (L.I > 2048) return false;                                              // h words per thread
    const FusedSmem s(L.H, L.E, L.I, k, bits);
    if (!s.aliases_fit(L.I)) return false;
    return s.total + 1024 <= 227 * 1024;
}

static size_t fused_smem(const moe_w4_layer& L) {
    return FusedSmem(L.H, L.E, L.I, L.top_k, code_bits_of(L)).total + 1024;
}

// Cooperative launch: every CTA resident at once (the exchanges wait on other
// CTAs); with programmatic dependent launch the prologue may overlap the
// previous kernel's tail.
static cudaLaunchConfig_t fused_config(const moe_w4_layer& L, cudaLaunchAttribute* attr, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((L.top_k + 1) * kPE);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = fused_smem(L);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cfg;
}

// The kernel's exchanges wait on other CTAs, so every CTA must be resident at
// once: the occupancy calculator's answer is checked (and cached per device and
// launch shape) before the fused path is taken, and the launch itself is
// cooperative.
bool decode_fused_supported(const moe_w4_layer& L) {
    if (!shape_ok(L)) return false;
    struct Entry { int dev, k; size_t smem; FusedKernel kern; bool ok; };
    static Entry cache[16] = {};
    static int ncache = 0;
    static std::mutex mu;   // first calls from several host threads fill the cache one at a time
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const size_t smem = fused_smem(L);
    const FusedKernel kern = fused_kernel_for(L);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].k == L.top_k && cache[i].smem == smem && cache[i].kern == kern)
            return cache[i].ok;
    bool ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess;
    if (ok) {
        int per_sm = 0, nsm = 0;
        ok = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFThreads, smem) == cudaSuccess &&
             cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
             per_sm * nsm >= (L.top_k + 1) * kPE;
    }
    cudaGetLastError();   // a refused query leaves no sticky error behind
    if (ncache < 16) cache[ncache++] = Entry{dev, L.top_k, smem, kern, ok};
    return ok;
}

// The six code tensor maps of a layer (routed and shared gate, up, down).
struct FusedMaps { CUtensorMap mg, mu, md, msg, msu, msd; };

static bool fused_maps(const moe_w4_layer& L, FusedMaps* m) {
    const int H = L.H, E = L.E, I = L.I, k = L.top_k;
    const int RG = I / kPE, DR = H / (kPE * k), b = code_bits_of(L);
    const uint32_t hbox = H * b / 1024 / kGuParts, dbox = I * b / 1024;   // box columns per copy
    return codes_map(&m->mg, L.gate.codes, (uint64_t)E * I, H, RG, hbox, b) &&
           codes_map(&m->mu, L.up.codes, (uint64_t)E * I, H, RG, hbox, b) &&
           codes_map(&m->md, L.down.codes, (uint64_t)E * H, I, DR, dbox, b) &&
           codes_map(&m->msg, L.sh_gate.codes, I, H, RG, hbox, b) &&
           codes_map(&m->msu, L.sh_up.codes, I, H, RG, hbox, b) &&
           codes_map(&m->msd, L.sh_down.codes, H, I, DR, dbox, b);
}

// One batch-1 call: x [H] -> out [H], routing into d.idx, d.w, d.gamma.
static cudaError_t launch_fused_row(const moe_w4_layer& L, const FusedMaps& m, const uint16_t* x, uint16_t* out,
                                    const DecodeWs& d, cudaStream_t st) {
    FusedArgs a{};
    a.x = x; a.router_w = L.router_w; a.router_bias = L.router_bias; a.shared_gate = L.shared_gate;
    a.gs = L.gate.scales; a.gb = L.gate.biases; a.us = L.up.scales; a.ub = L.up.biases;
    a.ds = L.down.scales; a.db = L.down.biases;
    a.sgs = L.sh_gate.scales; a.sgb = L.sh_gate.biases; a.sus = L.sh_up.scales; a.sub = L.sh_up.biases;
    a.sds = L.sh_down.scales; a.sdb = L.sh_down.biases;
    a.scores = d.fused_scores; a.hx = d.fused_hx; a.hsx = d.fused_hsx;
    a.idx_out = d.idx; a.w_out = d.w; a.gamma_out = d.gamma; a.out = out;
    a.ctrl = d.ctrl;
    a.H = L.H; a.E = L.E; a.I = L.I; a.k = L.top_k;
    cudaLaunchAttribute attr[2];
    const FusedKernel kern = fused_kernel_for(L);   // shared memory opt-in set by the support check
    cudaLaunchConfig_t cfg = fused_config(L, attr, st, true);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, m.mg, m.mu, m.md, m.msg, m.msu, m.msd);
    if (e != cudaSuccess) {   // refused with programmatic dependent launch: cooperative alone
        cudaGetLastError();
        cfg = fused_config(L, attr, st, false);
        e = cudaLaunchKernelEx(&cfg, kern, a, m.mg, m.mu, m.md, m.msg, m.msu, m.msd);
    }
    return e;
}

// Rows 0..T-1 one after another, each a complete batch-1 call on the stream
// (row t's routing at d.idx + t*k, d.w + t*k, d.gamma + t).  Consecutive calls
// overlap only through programmatic dependent launch, so each row still sees
// the exchange buffers as the previous row left them.  Returns the rows
// launched: fewer than T when a launch was refused or the tensor maps could
// not be built (0 then means nothing was launched).  Trace events: one before
// each row, then the rest after the last.
int launch_decode_fused_rows(const moe_w4_layer& L, int T, const uint16_t* x, uint16_t* out, const DecodeWs& d,
                             cudaStream_t st) {
    FusedMaps m;
    if (!fused_maps(L, &m)) return 0;
    const size_t k = (size_t)L.top_k, H = (size_t)L.H;
    for (int t = 0; t < T; ++t) {
        DecodeWs dt = d;
        dt.idx = d.idx + t * k;
        dt.w = d.w + t * k;
        dt.gamma = d.gamma + t;
        trace_mark(st, t);
        if (launch_fused_row(L, m, x + t * H, out + t * H, dt, st) != cudaSuccess) {
            cudaGetLastError();
            return t;
        }
    }
    trace_kernels(T);
    for (int i = T; i < T + 4; ++i) trace_mark(st, i);
    return T;
}

// Sizes of the fused kernel's exchange buffers (tagged 8-byte words) for a layer.
size_t fused_scores_bytes(const moe_w4_layer& L) { return (size_t)kScoreReplicas * 128 * L.top_k * 8; }
size_t fused_hx_bytes(const moe_w4_layer& L) { return (size_t)kHReplicas * (L.top_k + 1) * (L.I / 2) * 8; }
size_t fused_hsx_bytes(const moe_w4_layer& L) { return (size_t)kHReplicas * (L.top_k + 1) * (L.I / 16) * 2 * 8; }

}  // namespace mw4
