// Decode entry point for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: plugins inside an
// inference engine that owns all device memory and forbids allocation once it
// is serving, real-time loops that must never block on an allocator, or hosts
// whose memory plan is fixed before they learn the layer's shape.  For them,
// moe_w4_forward_decode_noalloc runs the same decode kernels as
// moe_w4_forward_decode, with the scratch those kernels need (partial router
// scores, selected experts and weights, the shared gate, the SwiGLU outputs and
// a small control header) placed in one file-scope device array of
// MOE_W4_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library keeps
// until the process exits.  Nothing on this path calls cudaMalloc, cudaFree or
// any allocating routine.
//
// In host code `g_noalloc_scratch` names a host-side stand-in, not the device
// array, so its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached; the first call on
// a device does this set-up.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mw4 {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_W4_NOALLOC_SCRATCH_BYTES];

static constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices] = {};
static std::atomic<int> g_noalloc_skip_publish{0};   // test hook (moe_w4_noalloc_test_skip_publish)
static std::mutex g_scratch_mu;   // first calls from several host threads set up the cache one at a time

static size_t up256n(size_t v) { return (v + 255) & ~size_t(255); }

// Compact decode-only layout inside the fixed array: control header, then the
// one-kernel T=1 decode's exchange buffers (router score partials, h, sums of
// h's pieces) at fixed offsets sized for the largest layer that kernel takes
// (top_k <= 8, I <= 2048), so that no call of another shape or layer ever writes there
// (the words there carry call tags that must only come from that kernel), then
// the buffers of the T >= 2 kernels: partial router scores, selected experts,
// weights, shared gate, SwiGLU outputs.
constexpr size_t kNoallocScoresBytes = 8 * 128 * 8 * 8;    // replicas x 128 k words, k <= 8
constexpr size_t kNoallocHxBytes = 8 * 9 * 1024 * 8;       // replicas x (k+1) * I/2 words
constexpr size_t kNoallocHsxBytes = 8 * 9 * 128 * 2 * 8;   // replicas x (k+1) * I/16 * 2 words
struct NoallocLayout { size_t ctrl, scores, hx, hsx, part, idx, w, gamma, hh, total; };

static NoallocLayout noalloc_layout(const moe_w4_layer& L, int T) {
    NoallocLayout n{};
    const size_t E = L.E, k = L.top_k, H = L.H, I = L.I, Tz = (size_t)T;
    const size_t nslice = (H + kRouterRowsPerCta - 1) / kRouterRowsPerCta;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += up256n(bytes); return at; };
    n.ctrl = take(sizeof(Ctrl));
    n.scores = take(kNoallocScoresBytes);
    n.hx = take(kNoallocHxBytes);
    n.hsx = take(kNoallocHsxBytes);
    n.part = take(nslice * Tz * E * 4);
    n.idx = take(Tz * k * 4);
    n.w = take(Tz * k * 4);
    n.gamma = take(Tz * 4);
    n.hh = take(Tz * (k + 1) * I * 4);
    n.total = o;
    return n;
}

// Device address of the scratch array on the current device (set-up on first use).
static cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace mw4

using namespace mw4;

extern "C" int moe_w4_forward_decode_noalloc(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out,
                                             cudaStream_t stream) {
    if (!L || L->E < 1 || L->top_k < 1 || L->top_k > 8 || L->top_k > L->E || L->H <= 0 || L->I <= 0)
        return MOE_W4_ERR_INVALID;
    if (L->H % kBM || L->I % kBM || L->H > 4096 || L->I > 4096 || L->E > 1024) return MOE_W4_ERR_UNSUPPORTED;
    if (L->code_bits != 0 && L->code_bits != 4 && L->code_bits != 8) return MOE_W4_ERR_UNSUPPORTED;
    if (L->code_format != MOE_W4_CODES_UINT && L->code_format != MOE_W4_CODES_E4M3) return MOE_W4_ERR_UNSUPPORTED;
    if (L->code_format == MOE_W4_CODES_E4M3 && L->code_bits != 8) return MOE_W4_ERR_UNSUPPORTED;
    if (T < 0) return MOE_W4_ERR_INVALID;
    if (T > kDecodeMaxT) return MOE_W4_ERR_UNSUPPORTED;
    if (T == 0) return MOE_W4_OK;
    // one-byte codes: only the one-kernel batch-1 decode, row by row (the
    // CUDA-core GEMVs of the fallback unpack nibbles)
    if (code_bits_of(*L) == 8 && !decode_fused_supported(*L)) return MOE_W4_ERR_UNSUPPORTED;
    if (!x || !out || !L->router_w || !L->shared_gate) return MOE_W4_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15) return MOE_W4_ERR_ALIGN;
    const moe_w4_mat* ms[6] = {&L->gate, &L->up, &L->down, &L->sh_gate, &L->sh_up, &L->sh_down};
    for (const moe_w4_mat* m : ms)
        if (!m->codes || !m->scales || !m->biases) return MOE_W4_ERR_INVALID;
    auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
    if (mis(L->router_w) || mis(L->shared_gate) || (L->router_bias && mis(L->router_bias))) return MOE_W4_ERR_ALIGN;
    for (const moe_w4_mat* m : ms)
        if (mis(m->codes) || mis(m->scales) || mis(m->biases)) return MOE_W4_ERR_ALIGN;
    const NoallocLayout n = noalloc_layout(*L, T);
    if (n.total > (size_t)MOE_W4_NOALLOC_SCRATCH_BYTES) return MOE_W4_ERR_SCRATCH;
    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_W4_ERR_LAUNCH;
    uint8_t* b = static_cast<uint8_t*>(base);
    // the completion counters must start at zero: clear the header every call, up to
    // the fused decode's call counter, which must keep counting (the exchange
    // buffers still hold earlier calls' tagged values)
    if (cudaMemsetAsync(b + n.ctrl, 0, offsetof(Ctrl, pad) + kCtrlEpochWord * sizeof(unsigned int), stream) !=
        cudaSuccess)
        return MOE_W4_ERR_LAUNCH;
    if (g_noalloc_skip_publish.load() &&   // failure-detection test hook: one CTA skips its router publish
        cudaMemsetAsync(b + n.ctrl + offsetof(Ctrl, pad) + kCtrlInjectWord * sizeof(unsigned int), 0x5A,
                        sizeof(unsigned int), stream) != cudaSuccess)
        return MOE_W4_ERR_LAUNCH;
    DecodeWs d{};
    d.part = reinterpret_cast<float*>(b + n.part);
    d.idx = reinterpret_cast<int32_t*>(b + n.idx);
    d.w = reinterpret_cast<float*>(b + n.w);
    d.gamma = reinterpret_cast<float*>(b + n.gamma);
    d.hh = reinterpret_cast<float*>(b + n.hh);
    d.counter = &reinterpret_cast<Ctrl*>(b + n.ctrl)->decode_counter;
    d.status = &reinterpret_cast<Ctrl*>(b + n.ctrl)->status;
    d.ctrl = reinterpret_cast<Ctrl*>(b + n.ctrl);
    d.fused_scores = reinterpret_cast<uint64_t*>(b + n.scores);
    d.fused_hx = reinterpret_cast<uint64_t*>(b + n.hx);
    d.fused_hsx = reinterpret_cast<uint64_t*>(b + n.hsx);
    return launch_decode(*L, T, x, out, d, stream) == cudaSuccess ? MOE_W4_OK : MOE_W4_ERR_LAUNCH;
}

// Copies the status word of the scratch array (the sticky MOE_W4_STATUS_* bits
// of the calls since the last one that cleared it) into caller memory.
extern "C" int moe_w4_noalloc_status(unsigned int* status, cudaStream_t stream) {
    if (!status) return MOE_W4_ERR_INVALID;
    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_W4_ERR_LAUNCH;
    const uint8_t* word = static_cast<const uint8_t*>(base) + offsetof(Ctrl, status);
    return cudaMemcpyAsync(status, word, sizeof(unsigned int), cudaMemcpyDefault, stream) == cudaSuccess
               ? MOE_W4_OK
               : MOE_W4_ERR_LAUNCH;
}

extern "C" int moe_w4_noalloc_test_skip_publish(int on) {
    g_noalloc_skip_publish.store(on ? 1 : 0);
    return MOE_W4_OK;
}
