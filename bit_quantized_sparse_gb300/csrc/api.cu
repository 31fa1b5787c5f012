// C ABI of libmoe_w4: argument validation, workspace layout and the three
// entry points (route, decode, prefill).  Everything is enqueued on the
// caller's stream; nothing here allocates, frees or synchronises.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "moe_w4_ablation.h"

namespace mw4 {

static cudaEvent_t* g_trace = nullptr;
static int g_ntrace = 0;
static int g_traced_kernels = 0;

void trace_mark(cudaStream_t st, int i) {
    if (!g_trace || i >= g_ntrace) return;
    // inside a stream capture the event becomes a graph node; outside it is a plain record
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(g_trace[i], st, cudaEventRecordExternal);
    else
        cudaEventRecord(g_trace[i], st);
}
void trace_kernels(int n) {
    if (g_trace) g_traced_kernels = n;
}

static size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

// Tile override: moe_w4_set_tile_override, else MOE_W4_FORCE_TILE (read once).
static std::atomic<int> g_tile_bn{0}, g_tile_du{0};
static std::once_flag g_tile_env_once;
static int set_tile(int bn, int du) {
    if (bn != 0 && bn != 32 && bn != 64 && bn != 128) return MOE_W4_ERR_INVALID;
    if (du != 0 && du != 1 && du != 2 && du != 4) return MOE_W4_ERR_INVALID;
    g_tile_bn.store(bn);
    g_tile_du.store(du);
    return MOE_W4_OK;
}
static void read_tile_env() {
    const char* v = std::getenv("MOE_W4_FORCE_TILE");
    if (!v) return;
    int bn = 0, du = 0;
    for (const char* p = v; *p;) {
        if (!std::strncmp(p, "bn=", 3)) bn = std::atoi(p + 3);
        else if (!std::strncmp(p, "du=", 3)) du = std::atoi(p + 3);
        const char* c = std::strchr(p, ',');
        if (!c) break;
        p = c + 1;
    }
    if (set_tile(bn, du) != MOE_W4_OK) std::fprintf(stderr, "moe_w4: MOE_W4_FORCE_TILE=%s ignored\n", v);
}

// Decode calls of up to this many rows run row by row through the fused
// batch-1 kernel, when it covers the layer; larger calls take the grouped path.
// The crossover, measured on the benchmark's layer (H=2048, E=256, top-8,
// I=512; CUDA-graph replays over 16 distinct layers, us per call):
//   rows           2    3    4    5    6    7    8
//   row by row    25   37   49   61   73   85   97
//   grouped       56   60   61   62   69   74   82
static std::atomic<int> g_fused_rows{kDecodeFusedRows};
int decode_fused_rows_max() { return g_fused_rows.load(); }

// Test hook (moe_w4_test_refuse_fused_after): at most this many rows of a call
// go through the one-kernel path before it behaves as if the next cooperative
// launch were refused; negative: off.
// (also used by the allocation-free decode in decode.cu)
static std::atomic<int> g_test_fused_allow{-1};
int test_fused_rows_allowed(int T) {
    const int a = g_test_fused_allow.load();
    return a < 0 || a > T ? T : a;
}

TileCfg tile_cfg(const moe_w4_layer& L, int T) {
    std::call_once(g_tile_env_once, read_tile_env);
    TileCfg c{kBN, (int64_t)T * L.top_k >= 64 * (int64_t)L.E ? down_blocks_per_unit(L.I) : 1};
    const int bn = g_tile_bn.load(), du = g_tile_du.load();
    if (bn) c.bn = bn;
    if (du && (du == 1 || L.I <= kDownReuseMaxI)) c.du = du;   // a reused tile keeps its whole K in TMEM
    return c;
}

WsLayout ws_layout(const moe_w4_layer& L, int T_max) {
    WsLayout w{};
    const size_t E = L.E, k = L.top_k, H = L.H, I = L.I;
    const size_t T = T_max < 1 ? 1 : (size_t)T_max;
    const size_t Td = T < (size_t)kDecodeMaxT ? T : (size_t)kDecodeMaxT;
    w.T_max = (int)T;
    w.nchunk_max = (int)((T + kChunk - 1) / kChunk);
    // blocks of kBN rows, or of as few as kMinBN under a tile override
    w.max_blocks = (int)((T * k + kMinBN - 1) / kMinBN + E + (T + kMinBN - 1) / kMinBN);
    w.max_tiles_gu = w.max_blocks * (int)(I / kBM);
    w.max_tiles_dn = w.max_blocks * (int)(H / kBM);
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += up256(bytes); return at; };
    w.ctrl = take(sizeof(Ctrl));
    w.logits = take(kRouterSplit * T * E * 4);   // partial router scores
    w.router_a = take((E + kBM - 1) / kBM * kBM * 3 * H * 2);
    w.x16 = take(T * H * 2);
    w.topk_idx = take(T * k * 4);
    w.topk_w = take(T * k * 4);
    w.gamma = take(T * 4);
    w.chunk_base = take((size_t)w.nchunk_max * E * 4);
    w.counts = take((E + 1) * 4);
    w.offsets = take((E + 2) * 4);
    w.perm = take(T * k * 4);
    w.inv = take(T * k * 4);
    w.blkinfo = take((size_t)w.max_blocks * sizeof(int4));
    w.unitinfo = take((size_t)w.max_blocks * sizeof(int4));
    w.ntiles = take(4 * sizeof(int32_t));
    w.hh = take((T * k + T) * I * 2);
    w.ys = take((T * k + T) * H * 2);
    const size_t nslice = (H + kRouterRowsPerCta - 1) / kRouterRowsPerCta;
    w.dec_part = take(nslice * Td * E * 4);
    w.dec_idx = take(Td * k * 4);
    w.dec_w = take(Td * k * 4);
    w.dec_gamma = take(Td * 4);
    w.dec_hh = take(Td * (k + 1) * I * 4);
    w.dec_scores = take(fused_scores_bytes(L));
    w.dec_hx = take(fused_hx_bytes(L));
    w.dec_hsx = take(fused_hsx_bytes(L));
    w.total = o;
    return w;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static int check_mat(const moe_w4_mat& m) {
    if (!m.codes || !m.scales || !m.biases) return MOE_W4_ERR_INVALID;
    if (!aligned16(m.codes) || !aligned16(m.scales) || !aligned16(m.biases)) return MOE_W4_ERR_ALIGN;
    return MOE_W4_OK;
}

static int check_layer(const moe_w4_layer* L) {
    if (!L) return MOE_W4_ERR_INVALID;
    if (L->E < 1 || L->top_k < 1 || L->top_k > 8 || L->top_k > L->E) return MOE_W4_ERR_INVALID;
    if (L->H <= 0 || L->I <= 0) return MOE_W4_ERR_INVALID;
    if (L->H % kBM || L->I % kBM || L->H > 4096 || L->I > 4096 || L->E > 1024) return MOE_W4_ERR_UNSUPPORTED;
    if (L->code_bits != 0 && L->code_bits != 4 && L->code_bits != 8) return MOE_W4_ERR_UNSUPPORTED;
    if (L->code_format != MOE_W4_CODES_UINT && L->code_format != MOE_W4_CODES_E4M3) return MOE_W4_ERR_UNSUPPORTED;
    if (L->code_format == MOE_W4_CODES_E4M3 && L->code_bits != 8) return MOE_W4_ERR_UNSUPPORTED;
    if (!L->router_w || !L->shared_gate) return MOE_W4_ERR_INVALID;
    if (!aligned16(L->router_w) || !aligned16(L->shared_gate) || (L->router_bias && !aligned16(L->router_bias)) ||
        (L->router_prep && !aligned16(L->router_prep)))
        return MOE_W4_ERR_ALIGN;
    const moe_w4_mat* ms[6] = {&L->gate, &L->up, &L->down, &L->sh_gate, &L->sh_up, &L->sh_down};
    for (const moe_w4_mat* m : ms) {
        const int r = check_mat(*m);
        if (r) return r;
    }
    return MOE_W4_OK;
}

// Fits calls of T tokens?  The layout is recomputed for the T the workspace
// was sized for: the largest T_max whose layout fits ws_bytes must be >= T.
static int check_ws(const moe_w4_layer& L, int T, const void* ws, size_t ws_bytes, WsLayout* out) {
    if (!ws) return MOE_W4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_W4_ERR_WORKSPACE;
    const WsLayout w = ws_layout(L, T);
    if (w.total > ws_bytes) return MOE_W4_ERR_WORKSPACE;
    *out = w;
    return MOE_W4_OK;
}

template <typename P>
static P* at(void* ws, size_t off) { return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off); }

// A failed launch returns MOE_W4_ERR_LAUNCH; with MOE_W4_DEBUG set in the
// environment the CUDA error string also goes to stderr.
static int launch_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_W4_OK;
    if (std::getenv("MOE_W4_DEBUG")) std::fprintf(stderr, "moe_w4: CUDA error %d: %s\n", (int)e, cudaGetErrorString(e));
    return MOE_W4_ERR_LAUNCH;
}

static RouteOut route_ws(void* ws, const WsLayout& w) {
    RouteOut o{};
    o.topk_idx = at<int32_t>(ws, w.topk_idx);
    o.topk_w = at<float>(ws, w.topk_w);
    o.gamma = at<float>(ws, w.gamma);
    o.counts = at<int32_t>(ws, w.counts);
    o.offsets = at<int32_t>(ws, w.offsets);
    o.perm = at<int32_t>(ws, w.perm);
    o.inv = at<int32_t>(ws, w.inv);
    o.chunk_base = at<int32_t>(ws, w.chunk_base);
    o.logits = at<float>(ws, w.logits);
    o.router_a = at<uint16_t>(ws, w.router_a);
    o.x16 = at<uint16_t>(ws, w.x16);
    o.blkinfo = at<int4>(ws, w.blkinfo);
    o.unitinfo = at<int4>(ws, w.unitinfo);
    o.ntiles = at<int32_t>(ws, w.ntiles);
    o.status = &at<Ctrl>(ws, w.ctrl)->status;
    return o;
}

}  // namespace mw4

using namespace mw4;

extern "C" {

size_t moe_w4_router_prep_bytes(const moe_w4_layer* L) {
    if (check_layer(L) != MOE_W4_OK) return 0;
    return router_prep_bytes(*L);
}

int moe_w4_prepare_router(const moe_w4_layer* L, void* dst, size_t dst_bytes, cudaStream_t stream) {
    const int r = check_layer(L);
    if (r) return r;
    if (!dst) return MOE_W4_ERR_INVALID;
    if (!aligned16(dst)) return MOE_W4_ERR_ALIGN;
    if (dst_bytes < router_prep_bytes(*L)) return MOE_W4_ERR_WORKSPACE;
    return launch_status(launch_router_prep(*L, static_cast<uint16_t*>(dst), stream));
}

size_t moe_w4_workspace_size(const moe_w4_layer* L, int T_max) {
    if (check_layer(L) != MOE_W4_OK || T_max < 0 || T_max > MOE_W4_MAX_TOKENS) return 0;
    return ws_layout(*L, T_max).total;
}

int moe_w4_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!workspace || ws_bytes < sizeof(Ctrl)) return MOE_W4_ERR_WORKSPACE;
    // the whole workspace: the fused decode's exchange buffers must start with no
    // call's tag in them
    return launch_status(cudaMemsetAsync(workspace, 0, ws_bytes, stream));
}

size_t moe_w4_status_offset(void) { return offsetof(Ctrl, status); }

int moe_w4_test_skip_publish(void* workspace, size_t ws_bytes, int on, cudaStream_t stream) {
    if (!workspace || ws_bytes < sizeof(Ctrl)) return MOE_W4_ERR_WORKSPACE;
    uint8_t* word = static_cast<uint8_t*>(workspace) + offsetof(Ctrl, pad) + kCtrlInjectWord * sizeof(unsigned int);
    return launch_status(cudaMemsetAsync(word, on ? 0x5A : 0, sizeof(unsigned int), stream));
}

int moe_w4_last_traced_kernels(void) { return g_traced_kernels; }

int moe_w4_test_block_records(const moe_w4_layer* L, int T, const void* workspace, size_t ws_bytes, int32_t* dst,
                              size_t dst_bytes, cudaStream_t stream) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 1 || !dst) return MOE_W4_ERR_INVALID;
    if (T > MOE_W4_MAX_TOKENS) return MOE_W4_ERR_UNSUPPORTED;
    WsLayout w;
    if ((r = check_ws(*L, T, const_cast<void*>(workspace), ws_bytes, &w))) return r;
    const size_t rec = (size_t)w.max_blocks * sizeof(int4);
    if (dst_bytes < 2 * sizeof(int32_t) + rec) return MOE_W4_ERR_WORKSPACE;
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    cudaError_t e = cudaMemcpyAsync(dst, ws + w.ntiles, 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst + 2, ws + w.blkinfo, rec, cudaMemcpyDeviceToDevice, stream);
    return launch_status(e);
}

size_t moe_w4_test_block_records_bytes(const moe_w4_layer* L, int T) {
    if (check_layer(L) != MOE_W4_OK || T < 1 || T > MOE_W4_MAX_TOKENS) return 0;
    return 2 * sizeof(int32_t) + (size_t)ws_layout(*L, T).max_blocks * sizeof(int4);
}

int moe_w4_set_tile_override(int bn, int du) {
    std::call_once(g_tile_env_once, read_tile_env);   // the environment first, so that this call wins
    return set_tile(bn, du);
}

int moe_w4_set_decode_fused_rows(int max_rows) {
    if (max_rows < 0 || max_rows > kDecodeMaxT) return MOE_W4_ERR_INVALID;
    g_fused_rows.store(max_rows ? max_rows : kDecodeFusedRows);
    return MOE_W4_OK;
}

int moe_w4_test_refuse_fused_after(int rows) {
    g_test_fused_allow.store(rows < 0 ? -1 : rows);
    return MOE_W4_OK;
}

int moe_w4_decode_path(const moe_w4_layer* L, int T, int* path) {
    int r = check_layer(L);
    if (r) return r;
    if (!path || T < 1) return MOE_W4_ERR_INVALID;
    if (T > kDecodeMaxT) return MOE_W4_ERR_UNSUPPORTED;
    *path = T <= decode_fused_rows_max() && decode_fused_supported(*L) ? MOE_W4_PATH_FUSED_ROWS : MOE_W4_PATH_GROUPED;
    return MOE_W4_OK;
}

int moe_w4_set_trace_events(cudaEvent_t* events, int n_events) {
    if (events && n_events < 1) return MOE_W4_ERR_INVALID;
    g_trace = events;
    g_ntrace = events ? n_events : 0;
    return MOE_W4_OK;
}

int moe_w4_route(const moe_w4_layer* L, int T, const moe_w4_bf16* x, int32_t* topk_idx, float* topk_w,
                 float* shared_gamma, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                 void* workspace, size_t ws_bytes, cudaStream_t stream) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 0) return MOE_W4_ERR_INVALID;
    if (T > MOE_W4_MAX_TOKENS) return MOE_W4_ERR_UNSUPPORTED;
    if (!topk_idx || !topk_w || !shared_gamma || !counts || !offsets || !perm || !inv)
        return MOE_W4_ERR_INVALID;
    if (T > 0 && !x) return MOE_W4_ERR_INVALID;
    if (T > 0 && !aligned16(x)) return MOE_W4_ERR_ALIGN;
    WsLayout w;
    if ((r = check_ws(*L, T, workspace, ws_bytes, &w))) return r;
    RouteOut o = route_ws(workspace, w);
    o.topk_idx = topk_idx; o.topk_w = topk_w; o.gamma = shared_gamma;
    o.counts = counts; o.offsets = offsets; o.perm = perm; o.inv = inv;
    o.blkinfo = nullptr; o.unitinfo = nullptr; o.x16 = nullptr;
    if (T == 0) {   // empty batch: zero counts and offsets, nothing else to write
        cudaMemsetAsync(counts, 0, (size_t)L->E * 4, stream);
        return launch_status(cudaMemsetAsync(offsets, 0, (size_t)(L->E + 1) * 4, stream));
    }
    cudaError_t e = launch_router_prefill(*L, T, x, o, stream);
    if (e == cudaSuccess) e = launch_grouping(*L, T, o, stream);
    return launch_status(e);
}

static int run_grouped(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out, void* workspace,
                       const WsLayout& w, cudaStream_t stream, int ablate = 0, void* scratch = nullptr);

int moe_w4_forward_decode(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out, void* workspace,
                          size_t ws_bytes, cudaStream_t stream) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 0 || T > kDecodeMaxT) return T < 0 ? MOE_W4_ERR_INVALID : MOE_W4_ERR_UNSUPPORTED;
    if (T == 0) return MOE_W4_OK;
    if (!x || !out) return MOE_W4_ERR_INVALID;
    if (!aligned16(x) || !aligned16(out)) return MOE_W4_ERR_ALIGN;
    WsLayout w;
    if ((r = check_ws(*L, T, workspace, ws_bytes, &w))) return r;
    // A few rows: one fused batch-1 kernel per row (each reads its 9 experts;
    // their latency, not their bytes, sets the time at these sizes).  More rows,
    // or a shape that kernel does not cover: the grouped path, which reads each
    // selected expert once for all the rows that chose it, on the tensor cores.
    if (T > decode_fused_rows_max() || !decode_fused_supported(*L))
        return run_grouped(L, T, x, out, workspace, w, stream);
    DecodeWs d{};
    d.part = at<float>(workspace, w.dec_part);
    d.idx = at<int32_t>(workspace, w.dec_idx);
    d.w = at<float>(workspace, w.dec_w);
    d.gamma = at<float>(workspace, w.dec_gamma);
    d.hh = at<float>(workspace, w.dec_hh);
    d.counter = &at<Ctrl>(workspace, w.ctrl)->decode_counter;
    d.status = &at<Ctrl>(workspace, w.ctrl)->status;
    d.ctrl = at<Ctrl>(workspace, w.ctrl);
    d.fused_scores = at<uint64_t>(workspace, w.dec_scores);
    d.fused_hx = at<uint64_t>(workspace, w.dec_hx);
    d.fused_hsx = at<uint64_t>(workspace, w.dec_hsx);
    const int done = launch_decode_fused_rows(*L, test_fused_rows_allowed(T), x, out, d, stream);
    if (done == T) return launch_status(cudaGetLastError());
    // a cooperative launch was refused (the grid cannot be resident at once on
    // this device or partition): the rows not yet enqueued take the grouped path
    const size_t H = (size_t)L->H;
    return run_grouped(L, T - done, x + done * H, out + done * H, workspace, w, stream);
}

// Routing, grouping and the grouped tensor-core GEMMs over T rows (the
// workspace checks already done).
static int run_grouped(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out, void* workspace,
                       const WsLayout& w, cudaStream_t stream, int ablate, void* scratch) {
    RouteOut o = route_ws(workspace, w);
    trace_mark(stream, 0);
    // measurement-only variants (moe_w4_ablation_prefill): the weights rebuilt in
    // fp16 by a separate pass first, read by the GEMMs with one-block down units
    const uint16_t* w16[6] = {};
    const TileCfg one_block{tile_cfg(*L, T).bn, 1};
    const bool sep = ablate == MOE_W4_ABLATE_SEPARATE_DEQUANT;
    cudaError_t e = sep ? launch_f16_weights(*L, static_cast<uint16_t*>(scratch), w16, o.status, stream) : cudaSuccess;
    if (e == cudaSuccess) e = launch_router_prefill(*L, T, x, o, stream);
    bool bad = false;
    if (e == cudaSuccess)
        e = ablate == MOE_W4_ABLATE_HOST_ROUTING ? host_grouping(*L, T, o, stream, &bad)
                                                  : launch_grouping(*L, T, o, stream, sep ? &one_block : nullptr);
    if (e != cudaSuccess) return MOE_W4_ERR_LAUNCH;
    if (bad) return MOE_W4_ERR_DEVICE;
    PrefillWs p{};
    p.blkinfo = o.blkinfo; p.unitinfo = o.unitinfo; p.ntiles = o.ntiles;
    p.offsets = o.offsets; p.perm = o.perm; p.inv = o.inv; p.topk_w = o.topk_w; p.gamma = o.gamma;
    p.x16 = o.x16;
    p.hh = at<uint16_t>(workspace, w.hh);
    p.ys = at<uint16_t>(workspace, w.ys);
    p.xg = p.ys;
    p.max_tiles_gu = w.max_tiles_gu;
    p.max_tiles_dn = w.max_tiles_dn;
    p.status = o.status;
    trace_kernels(7);
    return launch_status(launch_grouped_ffn(*L, T, x, out, p, stream, sep ? w16 : nullptr));
}


int moe_w4_forward_prefill(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out,
                           void* workspace, size_t ws_bytes, cudaStream_t stream) {
    int r = check_layer(L);
    if (r) return r;
    if (T < 0) return MOE_W4_ERR_INVALID;
    if (T > MOE_W4_MAX_TOKENS) return MOE_W4_ERR_UNSUPPORTED;
    if (T == 0) return MOE_W4_OK;
    if (!x || !out) return MOE_W4_ERR_INVALID;
    if (!aligned16(x) || !aligned16(out)) return MOE_W4_ERR_ALIGN;
    WsLayout w;
    if ((r = check_ws(*L, T, workspace, ws_bytes, &w))) return r;
    return run_grouped(L, T, x, out, workspace, w, stream);
}

size_t moe_w4_ablation_scratch_bytes(const moe_w4_layer* L, int mode) {
    if (check_layer(L) != MOE_W4_OK) return 0;
    return mode == MOE_W4_ABLATE_SEPARATE_DEQUANT ? f16_weights_bytes(*L) : 0;
}

int moe_w4_ablation_prefill(const moe_w4_layer* L, int T, const moe_w4_bf16* x, moe_w4_bf16* out, void* workspace,
                            size_t ws_bytes, int mode, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
    int r = check_layer(L);
    if (r) return r;
    if (mode != MOE_W4_ABLATE_HOST_ROUTING && mode != MOE_W4_ABLATE_SEPARATE_DEQUANT) return MOE_W4_ERR_INVALID;
    if (mode == MOE_W4_ABLATE_SEPARATE_DEQUANT) {
        if (!scratch) return MOE_W4_ERR_INVALID;
        if (!aligned16(scratch)) return MOE_W4_ERR_ALIGN;
        if (scratch_bytes < f16_weights_bytes(*L)) return MOE_W4_ERR_WORKSPACE;
    }
    if (T < 0) return MOE_W4_ERR_INVALID;
    if (T > MOE_W4_MAX_TOKENS) return MOE_W4_ERR_UNSUPPORTED;
    if (T == 0) return MOE_W4_OK;
    if (!x || !out) return MOE_W4_ERR_INVALID;
    if (!aligned16(x) || !aligned16(out)) return MOE_W4_ERR_ALIGN;
    WsLayout w;
    if ((r = check_ws(*L, T, workspace, ws_bytes, &w))) return r;
    return run_grouped(L, T, x, out, workspace, w, stream, mode, scratch);
}

const char* moe_w4_strerror(int status) {
    switch (status) {
        case MOE_W4_OK: return "ok";
        case MOE_W4_ERR_INVALID: return "invalid argument (NULL pointer, negative T or top_k out of range)";
        case MOE_W4_ERR_UNSUPPORTED: return "unsupported shape (H and I multiples of 128, H, I <= 4096, E <= 1024, decode T <= 16)";
        case MOE_W4_ERR_WORKSPACE: return "workspace missing, smaller than moe_w4_workspace_size or not 256-byte aligned";
        case MOE_W4_ERR_LAUNCH: return "a CUDA kernel launch failed";
        case MOE_W4_ERR_DEVICE: return "a kernel reported a device-side error in the status word";
        case MOE_W4_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case MOE_W4_ERR_SCRATCH:
            return "the call needs more scratch than the fixed MOE_W4_NOALLOC_SCRATCH_BYTES array of "
                   "moe_w4_forward_decode_noalloc";
        default: return "unknown status";
    }
}

}  // extern "C"
