// Device helpers shared by the kernels of libmoe_w4: inline PTX for mbarriers
// (every wait bounded), TMA bulk/tensor copies, cp.async, and the tcgen05
// tensor-core instructions (TMEM alloc, MMA, commit, loads).  sm_103a only.
#pragma once
#include <cfloat>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_w4.h"

#define MW4_DEV __device__ __forceinline__

namespace mw4 {

// ---------------------------------------------------------------------------
// status word (offset 0 of the workspace)
// ---------------------------------------------------------------------------
struct Ctrl {
    unsigned int status;          // sticky MOE_W4_STATUS_* bits
    unsigned int decode_counter;  // last-block-done counter of the decode router
    unsigned int pad[62];
};
static_assert(sizeof(Ctrl) == 256, "control header is 256 bytes");

// Release-ordered increment at GPU scope: after a CTA barrier, one thread's
// release makes the whole CTA's earlier writes visible to whoever acquires
// the counter (release ordering is cumulative over what the barrier ordered).
MW4_DEV unsigned int atomic_add_release_gpu(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Tagged values for cross-CTA exchanges: one 8-byte word, the float's bits in
// the low half and the writer's call tag in the high half, stored and loaded
// as single-copy-atomic 8-byte accesses at GPU scope.  A reader that sees its
// own call's tag has the value: the data is its own ready flag.
MW4_DEV void st_tagged(uint64_t* p, float v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(w) : "memory");
}
MW4_DEV uint64_t ld_tagged(const uint64_t* p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
MW4_DEV uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> 32); }
MW4_DEV float val_of(uint64_t w) { return __uint_as_float((uint32_t)w); }

MW4_DEV unsigned int atomic_add_acq_rel_gpu(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

MW4_DEV void raise_status(unsigned int* status, unsigned int bits) {
    if (status) atomicOr(status, bits);
}

// Debug builds (MW4_DEBUG_CHECKS, libmoe_w4_debug.so): an index read from the
// routing records (a position, a block or unit record) is checked against its
// range before use; out of range raises MOE_W4_STATUS_BAD_INDEX and the index
// is clamped into range, so the access stays inside its buffer.  In the
// product build the checks compile away.
MW4_DEV int checked_index(int v, int lo, int hi_excl, unsigned int* status) {
#ifdef MW4_DEBUG_CHECKS
    if (v < lo || v >= hi_excl) {
        raise_status(status, MOE_W4_STATUS_BAD_INDEX);
        return v < lo ? lo : hi_excl - 1;
    }
#else
    (void)lo; (void)hi_excl; (void)status;
#endif
    return v;
}

// ---------------------------------------------------------------------------
// shared-memory addresses
// ---------------------------------------------------------------------------
MW4_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
MW4_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
MW4_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MW4_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("{.reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0];}" :: "r"(smem_u32(bar)) : "memory");
}
MW4_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{.reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;}"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
MW4_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wall-clock bound for every wait: about two seconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
MW4_DEV uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase.  On timeout it raises
// MOE_W4_STATUS_WAIT_TIMEOUT, sets the CTA's abort flag and returns false.
// Any thread that sees the abort flag set also gives up at once.
// The waiting loop is out of line: it is the rare path, and single-pass kernels
// run from a cold instruction cache, where every inlined copy costs fetch time.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                   unsigned int* status) {
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            raise_status(status, MOE_W4_STATUS_WAIT_TIMEOUT);
            return false;
        }
    }
}
MW4_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned int* status) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, status);
}

// mbar_wait run by a whole converged warp; every lane gets lane 0's answer.
MW4_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned int* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag, status);
    return __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
}

// Programmatic dependent launch: wait until the preceding grid on the stream has
// completed and its memory is visible; let the next grid start launching.
MW4_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MW4_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// proxies and fences
// ---------------------------------------------------------------------------
// Generic-proxy writes to shared memory -> visible to the async proxy (TMA,
// tensor cores).  Executed by the writing threads before they signal.
MW4_DEV void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA and bulk copies (async proxy; completion counted in bytes on an mbarrier)
// ---------------------------------------------------------------------------
MW4_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
// Contiguous global -> shared copy; size and both addresses multiples of 16.
MW4_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
MW4_DEV void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16-byte, bypass L1)
// ---------------------------------------------------------------------------
MW4_DEV void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}
MW4_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MW4_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor-core MMA
// ---------------------------------------------------------------------------
// Allocation by one full warp; the TMEM base address is written to smem.
MW4_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MW4_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
MW4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MW4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored as rows of 128
// bytes (64 bf16) in the 128-byte swizzle pattern, 8-row atoms 1024 bytes
// apart.  `addr` must be 1024-byte aligned, plus 32 bytes per K=16 slice.
MW4_DEV uint64_t umma_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);          // start address
    d |= (uint64_t)(16 >> 4) << 16;                  // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: 8 rows * 128 B
    d |= (uint64_t)1 << 46;                          // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (format 0, both K-major),
// fp32 D.
MW4_DEV uint32_t umma_idesc_f16(int M, int N) {
    return (1u << 4)                     // D format fp32
         | (0u << 7)                     // A format fp16
         | (0u << 10)                    // B format fp16
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Instruction descriptor, kind::f16: bf16 A and B (format 1, both K-major),
// fp32 D.
MW4_DEV uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Warp-level issue: the whole (converged) warp executes these with the same
// operands and one elected lane issues the instruction.  Keeping the loop that
// feeds tcgen05.mma warp-uniform, rather than running it in one lane of a
// divergent branch, cuts the issue cost per MMA from about 44 cycles to about
// 12 on sm_103a (measured), which decides the rate for narrow N.  elect.sync
// elects the same lane every time for a full mask, so one thread issues both
// the MMAs and the commits that track them.
MW4_DEV void umma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{.reg .pred p, e; setp.ne.b32 p, %4, 0; elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
MW4_DEV void umma_f16_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{.reg .pred p, e; setp.ne.b32 p, %4, 0; elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
MW4_DEV void umma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{.reg .pred e; elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];}"
        :: "r"(smem_u32(bar)) : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns; thread t of the warp gets lane
// (base lane + t).  Must be followed by tmem_wait_ld before use.
MW4_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
MW4_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

MW4_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
MW4_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// 4-bit code unpacking to fp16 (exact), in "chunk order"
// ---------------------------------------------------------------------------
// A word holds the codes of 8 consecutive columns, n0 in the lowest nibble.
// fp16(1024) has a unit in the last place of 1, so a nibble OR-ed into bits
// 0..3 reads 1024 + q and one OR-ed into bits 4..7 reads 1024 + 16 q, both
// exactly.  One bitwise op therefore yields two columns; the four pairs come
// out as (n0,n4) (n1,n5) (n2,n6) (n3,n7), the second and fourth scaled by 16.
// The columns inside every 8-column chunk are thus stored in the order
//   kChunkOrder = {0, 4, 1, 5, 2, 6, 3, 7}
// and the other operand of the product (x, h) is stored in the same order.
MW4_DEV __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }
MW4_DEV uint32_t h2_as_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
MW4_DEV uint32_t bf162_as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

MW4_DEV int chunk_pos_of_col(int j) { return ((j & 3) << 1) | (j >> 2); }   // inverse of kChunkOrder
// 8-bit codes: two words per 8 columns, each giving the pairs (c0, c2), (c1, c3),
// so columns {0,2,1,3,4,6,5,7} sit at positions 0..7; position of column j.
MW4_DEV int chunk8_pos_of_col(int j) { return (j & 4) | ((j & 1) << 1) | ((j >> 1) & 1); }

// w = s*q + b for the four 8-bit codes of one word (lowest byte first): the fp16
// pairs (c0, c2) and (c1, c3).  1024 + q is exact in fp16 for q <= 255; each
// weight is rounded to fp16 once, in the fused multiply-add.
MW4_DEV void dequant4x8_f16(uint32_t w, __half2 s2, __half2 b2, uint32_t (&o)[2]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t p0 = (w & 0x00FF00FFu) | magic;           // 1024 + (q0, q2)
    const uint32_t p1 = ((w >> 8) & 0x00FF00FFu) | magic;    // 1024 + (q1, q3)
    const __half2 k1024 = u32_as_h2(magic);
    o[0] = h2_as_u32(__hfma2(s2, __hsub2(u32_as_h2(p0), k1024), b2));
    o[1] = h2_as_u32(__hfma2(s2, __hsub2(u32_as_h2(p1), k1024), b2));
}

// The four FP8 E4M3 codes of one word (lowest byte first) as fp16 pairs in the
// pair order of dequant4x8_f16: (c0, c2) and (c1, c3).  A byte permute puts c0,
// c2 in the low half-word and c1, c3 in the high one; each half-word converts
// to an fp16 pair (its upper byte to the upper half).  Every E4M3 value is
// exact in fp16.  dequant_e4m3x4_f16 then forms w = s*v + b, each weight
// rounded to fp16 once, in the fused multiply-add.
MW4_DEV void e4m3x4_to_f16(uint32_t w, uint32_t& v02, uint32_t& v13) {
    const uint32_t p = __byte_perm(w, 0u, 0x3120u);   // bytes c0, c2, c1, c3 (low to high)
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(v02), "=r"(v13) : "r"(p));
}

MW4_DEV void dequant_e4m3x4_f16(uint32_t w, __half2 s2, __half2 b2, uint32_t (&o)[2]) {
    uint32_t v0, v1;
    e4m3x4_to_f16(w, v0, v1);
    o[0] = h2_as_u32(__hfma2(s2, u32_as_h2(v0), b2));
    o[1] = h2_as_u32(__hfma2(s2, u32_as_h2(v1), b2));
}

// w = s*q + b for eight codes in chunk order; s2 = (s, s), s16 = (s/16, s/16),
// b2 = (b, b).  q (or 16 q) is recovered exactly and the product and sum are
// exact inside the fused multiply-add: each weight is rounded to fp16 once.
MW4_DEV void dequant8_f16(uint32_t w, __half2 s2, __half2 s16, __half2 b2, uint32_t (&o)[4]) {
    const uint32_t magic = 0x64006400u;
    const uint32_t w8 = w >> 8;
    const uint32_t p0 = (w & 0x000F000Fu) | magic;    // 1024 + (n0, n4)
    const uint32_t p1 = (w & 0x00F000F0u) | magic;    // 1024 + 16 (n1, n5)
    const uint32_t p2 = (w8 & 0x000F000Fu) | magic;   // 1024 + (n2, n6)
    const uint32_t p3 = (w8 & 0x00F000F0u) | magic;   // 1024 + 16 (n3, n7)
    const __half2 k1024 = u32_as_h2(magic);
    o[0] = h2_as_u32(__hfma2(s2, __hsub2(u32_as_h2(p0), k1024), b2));
    o[1] = h2_as_u32(__hfma2(s16, __hsub2(u32_as_h2(p1), k1024), b2));
    o[2] = h2_as_u32(__hfma2(s2, __hsub2(u32_as_h2(p2), k1024), b2));
    o[3] = h2_as_u32(__hfma2(s16, __hsub2(u32_as_h2(p3), k1024), b2));
}

MW4_DEV float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

MW4_DEV float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
// silu(z) = z sigmoid(z) = h + h tanh(h) with h = z/2: one hardware tanh
// (tanh.approx.f32, relative error about 2^-11, the size of the fp16 rounding the
// result then gets) instead of an exponential and a reciprocal, which halves the
// special-function work of the gate/up epilogue.
MW4_DEV float silu_tanh(float z) {
    const float h = 0.5f * z;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}


// ---------------------------------------------------------------------------
// warp-level selection (router)
// ---------------------------------------------------------------------------
// Order-preserving 32-bit key of a float: larger float, larger key.
MW4_DEV uint32_t order_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}

MW4_DEV void sort_desc_ce(uint64_t& a, uint64_t& b) {
    const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}

// Top-k (k <= 8) of E <= 32*NV (NV in 1, 2, 4, 8) scores in shared memory by one
// warp, larger score first and the lower expert index on equal scores.  Lane l
// holds experts l + 32 i as 64-bit words (order-preserving key << 32 | ~index),
// sorted once in descending order by a sorting network (19 exchanges for 8
// words), so a lane's best candidate is always its first word.  Each round takes
// the warp maximum of the keys (redux.sync), the lowest index holding it
// (redux.sync), and the lane that owns the winner drops its first word.  Absent
// experts (index >= E) carry key 0 and index 0xffffffff and sort last.  Lane
// r < k returns the r-th selection (index and score); with fewer than k experts
// the missing ones read -1.
template <int NV>
MW4_DEV void warp_topk_sorted(const float* sc, int E, int k, int& sel_idx, float& sel_val) {
    static_assert(NV == 1 || NV == 2 || NV == 4 || NV == 8, "sorting networks for 1, 2, 4 or 8 words");
    const int lane = threadIdx.x & 31;
    uint64_t c[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        c[i] = e < E ? ((uint64_t)order_key(sc[e]) << 32) | (uint32_t)~(uint32_t)e : 0ull;
    }
    // every branch compiles for every NV; indices are taken modulo NV so that the
    // branches of other widths stay in bounds (only the branch for this NV runs)
    if (NV == 2) sort_desc_ce(c[0], c[NV - 1]);
    if (NV == 4) {
        sort_desc_ce(c[0], c[1 % NV]); sort_desc_ce(c[2 % NV], c[3 % NV]);
        sort_desc_ce(c[0], c[2 % NV]); sort_desc_ce(c[1 % NV], c[3 % NV]);
        sort_desc_ce(c[1 % NV], c[2 % NV]);
    }
    if (NV == 8) {   // Batcher-style network, depth 6
        sort_desc_ce(c[0], c[2 % NV]); sort_desc_ce(c[1 % NV], c[3 % NV]);
        sort_desc_ce(c[4 % NV], c[6 % NV]); sort_desc_ce(c[5 % NV], c[7 % NV]);
        sort_desc_ce(c[0], c[4 % NV]); sort_desc_ce(c[1 % NV], c[5 % NV]);
        sort_desc_ce(c[2 % NV], c[6 % NV]); sort_desc_ce(c[3 % NV], c[7 % NV]);
        sort_desc_ce(c[0], c[1 % NV]); sort_desc_ce(c[2 % NV], c[3 % NV]);
        sort_desc_ce(c[4 % NV], c[5 % NV]); sort_desc_ce(c[6 % NV], c[7 % NV]);
        sort_desc_ce(c[2 % NV], c[4 % NV]); sort_desc_ce(c[3 % NV], c[5 % NV]);
        sort_desc_ce(c[1 % NV], c[4 % NV]); sort_desc_ce(c[3 % NV], c[6 % NV]);
        sort_desc_ce(c[1 % NV], c[2 % NV]); sort_desc_ce(c[3 % NV], c[4 % NV]); sort_desc_ce(c[5 % NV], c[6 % NV]);
    }
    sel_idx = -1;
    sel_val = 0.f;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        const uint32_t hk = (uint32_t)(c[0] >> 32), hix = ~(uint32_t)c[0];
        const uint32_t wmax = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t win = __reduce_min_sync(0xffffffffu, hk == wmax ? hix : 0xffffffffu);
        if (hix == win && win != 0xffffffffu) {
#pragma unroll
            for (int i = 0; i + 1 < NV; ++i) c[i] = c[i + 1];
            c[NV - 1] = 0ull;
        }
        if (lane == r && win < (uint32_t)E) { sel_idx = (int)win; sel_val = sc[win]; }
    }
}

// Top-k (k <= 8) of E <= 32*NV scores of one warp, larger score first and the
// lower expert index on equal scores; writes the experts by descending score
// and their softmax weights (over the selection, relative to the largest
// score).  NV <= 8 sorts each lane's candidates once (warp_topk_sorted); for
// larger NV each round takes the warp maximum (redux.sync) of the lanes' best
// remaining keys and, among the lanes holding it, the lowest expert index.
template <int NV>
MW4_DEV void select_topk_warp_n(const float* sc, int E, int k, int32_t* idx_out, float* w_out) {
    const int lane = threadIdx.x & 31;
    int mine = 0;
    float mval = 0.f;
    if (NV <= 8) {
        warp_topk_sorted<NV <= 8 ? NV : 8>(sc, E, k, mine, mval);
    } else {
        uint32_t key[NV];
        uint32_t live = 0;   // bit i: score lane + 32 i exists and is not taken
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            key[i] = e < E ? order_key(sc[e]) : 0u;
            if (e < E) live |= 1u << i;
        }
        for (int r = 0; r < k; ++r) {
            uint32_t bk = 0;
            int bi = 0x7fffffff;
            bool any = false;
#pragma unroll
            for (int i = 0; i < NV; ++i)   // ascending index in the lane: strict > keeps the lower one
                if (((live >> i) & 1u) && (!any || key[i] > bk)) { bk = key[i]; bi = lane + 32 * i; any = true; }
            const uint32_t wmax = __reduce_max_sync(0xffffffffu, any ? bk : 0u);
            const uint32_t win = __reduce_min_sync(0xffffffffu, (any && bk == wmax) ? (uint32_t)bi : 0xffffffffu);
            if ((int)(win & 31) == lane) live &= ~(1u << (win >> 5));
            if (lane == r) { mine = (int)win; mval = sc[win]; }
        }
    }
    const float v0 = __shfl_sync(0xffffffffu, mval, 0);
    const float ex = lane < k ? expf(mval - v0) : 0.f;
    float z = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (lane < k) {
        idx_out[lane] = mine;
        w_out[lane] = ex / z;
    }
}

// Selects the top-k of `sc` (E <= 1024 scores, owned by this warp), writes
// experts by descending score with softmax weights over the selection.
MW4_DEV void select_topk_warp(const float* sc, int E, int k, int32_t* idx_out, float* w_out) {
    if (E <= 32) select_topk_warp_n<1>(sc, E, k, idx_out, w_out);
    else if (E <= 64) select_topk_warp_n<2>(sc, E, k, idx_out, w_out);
    else if (E <= 128) select_topk_warp_n<4>(sc, E, k, idx_out, w_out);
    else if (E <= 256) select_topk_warp_n<8>(sc, E, k, idx_out, w_out);
    else if (E <= 512) select_topk_warp_n<16>(sc, E, k, idx_out, w_out);
    else select_topk_warp_n<32>(sc, E, k, idx_out, w_out);
}

MW4_DEV float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

}  // namespace mw4
