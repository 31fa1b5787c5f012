"""Benchmark of the W4 group-affine sparse-MoE layer on GB300.

Workload (one step): the long-prompt configuration -- a 16384-token prompt
processed as four 4096-row prefill chunks, then 64 consecutive batch-1 decode
steps; H=2048, E=256 experts, top-8, I=512, one shared expert, Zipf(1.2)-skewed
routing; every input seeded and synthetic.  The prefill chunks use one layer
(455 MB of packed weights, larger than L2).  The 64 decode steps cycle over 16
layers of the same shape with distinct weights (7.3 GB), as a multi-layer model
would, so a decode step never finds its layer's weights left in L2.

Printed (rank 0, one JSON line): whole-step tokens/s, prefill and decode
tokens/s, the roofline of the dominant kernel and of the decode step, the CPU
oracle timed on this host, the end-to-end rate through host buffers, clocks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4g64 MoE layer tok/s at T=1 & T=4096; % of HBM / bf16 TC roofline"
WORKLOAD = "long_T16384"
N_REPLICAS = 16
PREFILL_KERNELS = ["router_scores", "topk", "group", "gather_rows", "gemm_gate_up", "gemm_down", "combine"]
DECODE_KERNELS = ["decode_router", "decode_gate_up", "decode_down"]   # the three-kernel path
DECODE_FUSED = ["decode_fused"]
SMALL_T = (2, 4, 6, 8)   # multi-row decode batches measured beside the step
MULTIROW_PATHS = {1: "one-kernel batch-1 decode once per row (decode_fused_kernel, T launches)",
                  2: "grouped tensor-core path (one read per selected expert)"}
# prefill tile choices of the ablation table: (token rows per block, row blocks per down unit); the first is the default
TILE_CHOICES = ((128, 4), (128, 2), (128, 1), (64, 4), (64, 2), (64, 1), (32, 1))
ABLATION_T = (512, 2048, 4096)   # prefill sizes of the ablations (2048 rows = 16,384 assignments, 64 per expert)
CPU_SAMPLE = (8192, 32)   # oracle sample for cpu_baseline: prefill rows, decode rows
W8_REPLICAS = 8    # distinct one-byte-code layers each format-variant decode measurement cycles
# weight codes: (bits, code_format) -- unsigned 4-bit, unsigned 8-bit, FP8 E4M3
CODES = {"u4": (4, 0), "u8": (8, 0), "e4m3": (8, 1)}
VARIANTS = ("u8", "e4m3")   # format variants measured beside the step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["step", "prefill_chunk", "decode"], default="step",
                    help="step: the timed benchmark; prefill_chunk / decode: run --calls plain library calls on "
                         "one layer of the workload and exit (for profilers)")
    ap.add_argument("--calls", type=int, default=2)
    ap.add_argument("--codes", choices=list(CODES), default="u4",
                    help="weight codes of the layer a --case run uses")
    ap.add_argument("--no-multirow", action="store_true",
                    help="skip the multi-row decode measurement (for launch lists that should hold the step's "
                         "kernels only)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the 8-bit weight-format measurement (for launch lists of the step's kernels only)")
    ap.add_argument("--ablations", action="store_true",
                    help="also measure the prefill design choices against their alternatives (tile table, "
                         "host-synchronised routing, router weights split per call); adds an 'ablations' object")
    return ap.parse_args()


def run_case(args):
    """Small untimed runs for profilers: one layer, `calls` library calls."""
    import torch
    from bit_quantized_sparse_gb300 import moe_w4 as mw
    from bit_quantized_sparse_gb300 import synthetic as S
    c = S.CONFIGS[WORKLOAD]
    T = c["chunk"] if args.case == "prefill_chunk" else 1
    L0, x = S.draw_config(WORKLOAD, T=T)
    xd = mw.tokens_to_device(x)
    bits, fmt = CODES[args.codes]
    dl = mw.DeviceLayer(L0 if args.codes == "u4" else
                        S.draw_layer_torch(c["H"], c["E"], c["I"], c["top_k"], c["zipf"], seed=2000, bits=bits,
                                           fmt=fmt))
    for _ in range(args.calls):
        (mw.forward_prefill if args.case == "prefill_chunk" else mw.forward_decode)(dl, xd)
    torch.cuda.synchronize()
    if dl.status() != 0:
        raise RuntimeError(f"device status {dl.status()}")
    print(json.dumps({"case": args.case, "codes": args.codes, "calls": args.calls, "T": T, "ok": True}))


# ---------------------------------------------------------------------------
# multi-process plumbing (one process per GPU; replicas, no data-path exchange)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_max(value, dist, device):
    """Max over ranks of a float (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, world, seconds):
    """Whole-job throughput: every rank processes the same units (weak scaling)."""
    return units_per_rank * world / seconds


# ---------------------------------------------------------------------------
# measured peaks and clocks
# ---------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu figures
    (profiles/traffic.json), or None when the kernel's source files have changed
    since that capture (their sha256 no longer matches) or it was never captured."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    for e in json.load(open(path))["kernels"]:
        if e["kernel"] != kernel:
            continue
        h = hashlib.sha256()
        for f in e["sources"]:
            fp = os.path.join(ROOT, "bit_quantized_sparse_gb300", f)
            if not os.path.exists(fp):
                return None
            h.update(open(fp, "rb").read())
        return int(e["dram_bytes_per_launch"]) if h.hexdigest() == e["sha256"] else None
    return None


class ClockSampler:
    """nvidia-smi sampled every 20 ms while the timed regions run."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def build_workload(torch, mw, S, device):
    c = S.CONFIGS[WORKLOAD]
    L0, x = S.draw_config(WORKLOAD)
    xdec = S.draw_tokens(L0, c["decode_steps"], c["seed"], stream=1)
    layers = [mw.DeviceLayer(L0, device)]
    for r in range(1, N_REPLICAS):
        Lr = S.draw_layer_torch(c["H"], c["E"], c["I"], c["top_k"], c["zipf"], seed=1000 + r, device=device)
        layers.append(mw.DeviceLayer(Lr, device))
    return c, L0, x, xdec, layers


def run_gpu(args, rank, local_rank, world, dist):
    import torch
    from bit_quantized_sparse_gb300 import moe_w4 as mw
    from bit_quantized_sparse_gb300 import synthetic as S

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    c, L0, x_np, xdec_np, layers = build_workload(torch, mw, S, device)
    T, chunk, ndec, H = c["T"], c["chunk"], c["decode_steps"], c["H"]
    x = mw.tokens_to_device(x_np, device)
    xdec = mw.tokens_to_device(xdec_np, device)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    outdec = torch.empty((ndec, H), dtype=torch.bfloat16, device=device)
    ws = layers[0].workspace(chunk)
    stream = torch.cuda.Stream(device)

    def prefill_part():
        for i in range(0, T, chunk):
            mw.forward_prefill(layers[0], x[i:i + chunk], out=out[i:i + chunk], ws=ws)

    def decode_part():
        for i in range(ndec):
            mw._check(mw.moe_w4_forward_decode(ctypes.byref(layers[i % N_REPLICAS].c), 1, xdec[i:i + 1].data_ptr(),
                                               outdec[i:i + 1].data_ptr(), ws.data_ptr(), ws.numel(),
                                               torch.cuda.current_stream().cuda_stream), "decode")

    def step():
        prefill_part()
        decode_part()

    # eager warm-up (first-call host set-up happens outside any capture)
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    if layers[0].status() != 0:
        raise RuntimeError(f"device status {layers[0].status()} after warm-up")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    g_step, g_pre, g_dec = capture(step), capture(prefill_part), capture(decode_part)

    def timed(g, n, per=None):
        """Seconds for n replays of g (max over ranks), events on the replay stream
        around each replay; `per`, if given, receives each replay's seconds."""
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for i in range(n):
                g.replay()
                evs[i + 1].record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        if per is not None:
            per.extend(evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(n))
        return reduce_max(evs[0].elapsed_time(evs[n]) / 1e3, dist, device)

    clk = ClockSampler(local_rank).__enter__()   # sampling spans every timed region of the run
    per_step, per_pre, per_dec = [], [], []
    t_step = timed(g_step, args.steps, per_step)
    t_pre = timed(g_pre, args.steps, per_pre)
    t_dec = timed(g_dec, args.steps, per_dec)

    # multi-row decode (T = 2, 4 and 8 rows per call): calls cycling the replica
    # layers over slices of the decode rows; the bytes a call must move count
    # every distinct expert its rows select once (routing by the library's own
    # router).  Each size is also timed on the path the library did not choose
    # (the row limit of moe_w4_set_decode_fused_rows moved past it), which is
    # the measurement behind that limit.
    small = {}
    n_small = 32

    def time_small(Tm):
        def dec_small():
            for i in range(n_small):
                o = (i * Tm) % (ndec - ndec % Tm)   # whole slices of Tm rows inside the decode rows
                mw._check(mw.moe_w4_forward_decode(ctypes.byref(layers[i % N_REPLICAS].c), Tm,
                                                   xdec[o:o + Tm].data_ptr(), outdec[o:o + Tm].data_ptr(),
                                                   ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream),
                          "decode T>1")
        with torch.cuda.stream(stream):
            dec_small()
        torch.cuda.synchronize()
        return timed(capture(dec_small), args.steps) / args.steps / n_small

    for Tm in (() if args.no_multirow else SMALL_T):
        t_small = time_small(Tm)
        path = mw.decode_path(layers[0], Tm)
        t_alt = None
        if mw.decode_path(layers[0], 1) == mw.MOE_W4_PATH_FUSED_ROWS:   # both paths exist for this layer
            mw._check(mw.moe_w4_set_decode_fused_rows(1 if path == mw.MOE_W4_PATH_FUSED_ROWS else mw.DECODE_MAX_T),
                      "row limit")
            try:
                t_alt = time_small(Tm)
            finally:
                mw._check(mw.moe_w4_set_decode_fused_rows(0), "row limit")
        distinct = []
        for i in range(n_small):
            o = (i * Tm) % (ndec - ndec % Tm)   # whole slices of Tm rows inside the decode rows
            cnt = mw.route(layers[i % N_REPLICAS], xdec[o:o + Tm])["counts"]
            distinct.append(int((cnt > 0).sum().item()))
        small[Tm] = (t_small, float(np.mean(distinct)), path, t_alt)

    # per-kernel durations: the library records events around its kernels
    def traced(fn, names):
        n = len(names) + 1
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        with torch.cuda.stream(stream):
            for e in evs:
                e.record(stream)
        torch.cuda.synchronize()
        arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
        mw._check(mw.moe_w4_set_trace_events(arr, n), "trace")
        try:
            g = capture(fn)
            nk = mw.moe_w4_last_traced_kernels()
        finally:
            mw.moe_w4_set_trace_events(None, 0)
        acc = np.zeros(n - 1)
        for _ in range(args.warmup):
            g.replay()
        for _ in range(args.steps):
            g.replay()
            torch.cuda.synchronize()
            acc += [evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(n - 1)]
        return dict(zip(names[:nk], (acc[:nk] / args.steps).tolist()))

    xc = x[:chunk]
    k_pre = traced(lambda: mw.forward_prefill(layers[0], xc, out=out[:chunk], ws=ws), PREFILL_KERNELS)
    k_dec = traced(lambda: mw._check(mw.moe_w4_forward_decode(
        ctypes.byref(layers[1].c), 1, xdec[:1].data_ptr(), outdec[:1].data_ptr(), ws.data_ptr(), ws.numel(),
        torch.cuda.current_stream().cuda_stream), "decode"), DECODE_KERNELS)
    if len(k_dec) == 1:                     # batch-1 decode of this shape is one fused kernel
        k_dec = {DECODE_FUSED[0]: next(iter(k_dec.values()))}
    # a multi-row decode call (4 rows): where its time goes (one fused kernel per
    # row, or the grouped path's kernels)
    names4 = ([f"decode_fused_row{i}" for i in range(4)]
              if mw.decode_path(layers[1], 4) == mw.MOE_W4_PATH_FUSED_ROWS else PREFILL_KERNELS)
    k_dec4 = {} if args.no_multirow else traced(lambda: mw._check(mw.moe_w4_forward_decode(
        ctypes.byref(layers[1].c), 4, xdec[:4].data_ptr(), outdec[:4].data_ptr(), ws.data_ptr(), ws.numel(),
        torch.cuda.current_stream().cuda_stream), "decode T=4"), names4)

    # weight-format variants (8-bit affine codes, FP8 E4M3 codes): layers of the
    # same shape with one-byte codes; a 4096-row prefill chunk and batch-1
    # decode calls cycling W8_REPLICAS distinct layers (6.8 GB, far above L2)
    variants = {}
    for vname in (() if args.no_variants else VARIANTS):
        bits, fmt = CODES[vname]
        l8 = [mw.DeviceLayer(S.draw_layer_torch(c["H"], c["E"], c["I"], c["top_k"], c["zipf"], seed=2000 + r,
                                                device=device, bits=bits, fmt=fmt), device)
              for r in range(W8_REPLICAS)]
        ws8 = l8[0].workspace(chunk)

        def pre8():
            mw.forward_prefill(l8[0], xc, out=out[:chunk], ws=ws8)

        def dec8():
            for i in range(n_small):
                mw._check(mw.moe_w4_forward_decode(ctypes.byref(l8[i % W8_REPLICAS].c), 1, xdec[i:i + 1].data_ptr(),
                                                   outdec[i:i + 1].data_ptr(), ws8.data_ptr(), ws8.numel(),
                                                   torch.cuda.current_stream().cuda_stream), "decode " + vname)
        with torch.cuda.stream(stream):
            pre8()
            dec8()
        torch.cuda.synchronize()
        if l8[0].status() != 0:
            raise RuntimeError(f"device status {l8[0].status()} ({vname} layer)")
        t8_pre = timed(capture(pre8), args.steps) / args.steps
        t8_dec = timed(capture(dec8), args.steps) / args.steps / n_small
        k8_pre = traced(pre8, PREFILL_KERNELS)
        variants[vname] = dict(t_pre=t8_pre, t_dec=t8_dec, k_pre=k8_pre, bits=bits)
        del l8, ws8

    abl = run_ablations(torch, mw, c, layers[0], x, out, ws, stream, timed, capture, args) if args.ablations else None

    # end to end through host buffers, every step: the step's inputs are copied in
    # from pinned host memory and its outputs copied back, segment by segment (the
    # four 4096-row prefill chunks, then the decode rows).  A segment's rows go in
    # on one copy stream, the segment runs once they are in, and its output goes
    # out on a second copy stream while the next segment runs.  Events order the
    # reuse of a device buffer across steps: its copy-in waits for the previous
    # step's compute on it, and the compute that overwrites an output waits for
    # the previous step's copy-out.
    x_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    xd_host = torch.empty((ndec, H), dtype=torch.bfloat16, pin_memory=True)
    xd_host.copy_(xdec.cpu())
    o_host = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    od_host = torch.empty((ndec, H), dtype=torch.bfloat16, pin_memory=True)
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    starts = list(range(0, T, chunk))
    g_seg = [capture(lambda i=i: mw.forward_prefill(layers[0], x[i:i + chunk], out=out[i:i + chunk], ws=ws))
             for i in starts] + [g_dec]
    seg_in = [(x[i:i + chunk], x_host[i:i + chunk]) for i in starts] + [(xdec, xd_host)]
    seg_out = [(o_host[i:i + chunk], out[i:i + chunk]) for i in starts] + [(od_host, outdec)]
    done_read = [None] * len(g_seg)   # compute finished with the segment's input
    done_out = [None] * len(g_seg)    # copy-out of the segment's output finished

    def e2e_steps(n):
        for _ in range(n):
            arrived = []
            for sgi, (dst, src) in enumerate(seg_in):
                with torch.cuda.stream(h2d):
                    if done_read[sgi] is not None:
                        h2d.wait_event(done_read[sgi])
                    dst.copy_(src, non_blocking=True)
                    arrived.append(torch.cuda.Event())
                    arrived[-1].record(h2d)
            for sgi, g in enumerate(g_seg):
                with torch.cuda.stream(stream):
                    stream.wait_event(arrived[sgi])
                    if done_out[sgi] is not None:
                        stream.wait_event(done_out[sgi])
                    g.replay()
                    done_read[sgi] = torch.cuda.Event()
                    done_read[sgi].record(stream)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(done_read[sgi])
                    seg_out[sgi][0].copy_(seg_out[sgi][1], non_blocking=True)
                    done_out[sgi] = torch.cuda.Event()
                    done_out[sgi].record(d2h)

    e2e_steps(args.warmup)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_steps(args.steps)
    torch.cuda.synchronize()
    t_e2e = reduce_max(time.perf_counter() - t0, dist, device)
    clk.__exit__(None, None, None)
    clocks = clk.summary()
    status = layers[0].status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    return dict(c=c, L0=L0, x_np=x_np, xdec_np=xdec_np, t_step=t_step, t_pre=t_pre, t_dec=t_dec, t_e2e=t_e2e, small=small,
                per_step=per_step, per_pre=per_pre, per_dec=per_dec,
                variants=variants, clocks=clocks, k_pre=k_pre, k_dec=k_dec, k_dec4=k_dec4,
                gpu=torch.cuda.get_device_name(device),
                ablations=abl)


def run_ablations(torch, mw, c, dl, x, out, ws, stream, timed, capture, args):
    """The prefill's design choices against their alternatives, on the
    workload's first layer and the first T rows of its prompt:
    - tiles: ms per call for each (token rows per block, row blocks per down
      unit) of TILE_CHOICES (CUDA-graph replays, like the step);
    - routing: ms per call, eager calls, with the GPU-resident grouping and with
      the host-synchronised one (moe_w4_ablation_prefill);
    - router_prep: ms per call (graph replays) with the router weights prepared
      once and split on every call;
    - dequant: ms per call (graph replays) with the weights rebuilt in the
      GEMMs' tiles (the product) and with a separate pass that writes every
      weight in fp16 before the GEMMs read them back;
    - paired: each alternative against the product path in alternating
      rounds, with the median ratio and its bootstrap confidence interval."""
    res = {"tiles_ms": {}, "routing_ms": {}, "router_prep_ms": {}, "dequant_ms": {}}
    nscr = mw.moe_w4_ablation_scratch_bytes(ctypes.byref(dl.c), mw.MOE_W4_ABLATE_SEPARATE_DEQUANT)
    scratch = torch.empty(nscr, dtype=torch.uint8, device=x.device)   # every weight in fp16 (1.6 GB)
    st = lambda: torch.cuda.current_stream().cuda_stream

    def graph_ms(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        return 1e3 * timed(capture(fn), args.steps) / args.steps

    def eager_ms(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            torch.cuda.synchronize()
        return 1e3 * (time.perf_counter() - t0) / n

    def paired_graphs(fa, fb, rounds):
        """A and B captured as graphs, then replayed in alternating rounds (A
        first in even rounds, B first in odd ones), each replay between its own
        events on the replay stream."""
        gs = []
        for fn in (fa, fb):
            with torch.cuda.stream(stream):
                fn()
            torch.cuda.synchronize()
            gs.append(capture(fn))
        for g in gs:
            for _ in range(args.warmup):
                g.replay()
        torch.cuda.synchronize()
        ts = ([], [])
        for i in range(rounds):
            for j in ((0, 1) if i % 2 == 0 else (1, 0)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    gs[j].replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                ts[j].append(e0.elapsed_time(e1) / 1e3)
        return paired_ratio(*ts)

    def paired_eager(fa, fb, rounds):
        """The same with eager calls (host wall clock, synchronised per call)."""
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fa()
                fb()
            torch.cuda.synchronize()
            ts = ([], [])
            for i in range(rounds):
                for j in ((0, 1) if i % 2 == 0 else (1, 0)):
                    t0 = time.perf_counter()
                    (fa, fb)[j]()
                    torch.cuda.synchronize()
                    ts[j].append(time.perf_counter() - t0)
        return paired_ratio(*ts)

    plain = mw.MoeW4Layer.from_buffer_copy(dl.c)
    plain.router_prep = None
    res["paired"] = {}
    rounds = max(2 * args.steps, 20)
    for Tm in ABLATION_T:
        xs, os_ = x[:Tm], out[:Tm]
        row = {}
        try:
            for bn, du in TILE_CHOICES:
                assert mw.moe_w4_set_tile_override(bn, du) == mw.MOE_W4_OK
                row[f"bn{bn}_du{du}"] = graph_ms(lambda: mw.forward_prefill(dl, xs, out=os_, ws=ws))
        finally:
            mw.moe_w4_set_tile_override(0, 0)
        res["tiles_ms"][f"T{Tm}"] = row

        def host_routed():
            mw._check(mw.moe_w4_ablation_prefill(ctypes.byref(dl.c), Tm, xs.data_ptr(), os_.data_ptr(), ws.data_ptr(),
                                                 ws.numel(), mw.MOE_W4_ABLATE_HOST_ROUTING, None, 0, st()), "ablation")

        def separate_dequant():
            mw._check(mw.moe_w4_ablation_prefill(ctypes.byref(dl.c), Tm, xs.data_ptr(), os_.data_ptr(), ws.data_ptr(),
                                                 ws.numel(), mw.MOE_W4_ABLATE_SEPARATE_DEQUANT, scratch.data_ptr(),
                                                 scratch.numel(), st()), "ablation")
        res["dequant_ms"][f"T{Tm}"] = {"fused_in_gemm": row[f"bn{TILE_CHOICES[0][0]}_du{TILE_CHOICES[0][1]}"],
                                      "separate_fp16_pass": graph_ms(separate_dequant)}
        n = max(args.steps, 5)
        res["routing_ms"][f"T{Tm}"] = {
            "gpu_resident_eager": eager_ms(lambda: mw.forward_prefill(dl, xs, out=os_, ws=ws), n),
            "host_synchronised_eager": eager_ms(host_routed, n),
            "gpu_resident_graph": graph_ms(lambda: mw.forward_prefill(dl, xs, out=os_, ws=ws))}

        def split_each_call():
            mw._check(mw.moe_w4_forward_prefill(ctypes.byref(plain), Tm, xs.data_ptr(), os_.data_ptr(), ws.data_ptr(),
                                                ws.numel(), st()), "prefill")
        res["router_prep_ms"][f"T{Tm}"] = {"prepared_once": row[f"bn{TILE_CHOICES[0][0]}_du{TILE_CHOICES[0][1]}"],
                                          "split_every_call": graph_ms(split_each_call)}

        # the same comparisons as paired, interleaved rounds: A is always the product path
        def product():
            mw.forward_prefill(dl, xs, out=os_, ws=ws)

        def bn64():
            assert mw.moe_w4_set_tile_override(64, 0) == mw.MOE_W4_OK
            try:
                mw.forward_prefill(dl, xs, out=os_, ws=ws)
            finally:
                mw.moe_w4_set_tile_override(0, 0)
        res["paired"][f"T{Tm}"] = {
            "separate_fp16_pass_vs_fused": paired_graphs(product, separate_dequant, rounds),
            "host_synchronised_vs_gpu_resident_eager": paired_eager(product, host_routed, rounds),
            "split_every_call_vs_prepared_once": paired_graphs(product, split_each_call, rounds),
            "bn64_vs_default_tile": paired_graphs(product, bn64, rounds)}
    if dl.status() != 0:
        raise RuntimeError(f"device status {dl.status()} after the ablations")
    return res


# ---------------------------------------------------------------------------
# algorithmic work (per unit) for the roofline
# ---------------------------------------------------------------------------
def expert_bytes(H, I, bits=4):
    """Packed codes plus a bf16 scale and bias per 64 weights, for gate, up and down."""
    w = 3 * H * I
    return w * bits // 8 + 2 * 2 * (w // 64)


def decode_bytes_rows(c, T, distinct):
    """Bytes a decode call of T rows must move: each distinct selected expert
    once, the shared expert, router weights, shared gate, x and out."""
    H, E, I = c["H"], c["E"], c["I"]
    return (distinct + 1) * expert_bytes(H, I) + H * E * 4 + H * 4 + T * H * 2 + T * H * 2


def decode_bytes(c, T=1, bits=4):
    """Bytes one decode call must move: k+1 experts' packed weights, router
    weights, shared gate, x and out."""
    H, E, I, k = c["H"], c["E"], c["I"], c["top_k"]
    return (k + 1) * expert_bytes(H, I, bits) + H * E * 4 + H * 4 + T * H * 2 + T * H * 2


def gemm_flops(c, T, which):
    H, I, k = c["H"], c["I"], c["top_k"]
    rows = T * k + T
    return 2 * rows * H * 2 * I if which == "gate_up" else 2 * rows * I * H


def spread(values, scale=1.0, n_boot=2000, seed=0):
    """Median, 10th and 90th percentile of per-replay times (seconds), scaled,
    and a 95% bootstrap confidence interval of the median (percentile method,
    n_boot resamples of the replays with replacement, seeded)."""
    if not values:
        return None
    v = np.sort(np.asarray(values, np.float64)) * scale
    rng = np.random.default_rng(seed)
    meds = np.median(v[rng.integers(0, v.size, size=(n_boot, v.size))], axis=1)
    return {"median": float(np.median(v)), "p10": float(np.percentile(v, 10)), "p90": float(np.percentile(v, 90)),
            "median_ci95": [float(np.percentile(meds, 2.5)), float(np.percentile(meds, 97.5))],
            "replays": int(v.size)}


def paired_ratio(a_s, b_s, n_boot=2000, seed=0):
    """Paired comparison of two implementations timed in alternating rounds
    (per-round seconds of A and of B, same length): the median of each in ms,
    and the median of the per-round ratios B/A with a 95% bootstrap confidence
    interval (percentile method, rounds resampled with replacement, seeded)."""
    a = np.asarray(a_s, np.float64)
    b = np.asarray(b_s, np.float64)
    r = b / a
    rng = np.random.default_rng(seed)
    meds = np.median(r[rng.integers(0, r.size, size=(n_boot, r.size))], axis=1)
    return {"a_ms": 1e3 * float(np.median(a)), "b_ms": 1e3 * float(np.median(b)),
            "ratio_median": float(np.median(r)),
            "ratio_ci95": [float(np.percentile(meds, 2.5)), float(np.percentile(meds, 97.5))], "rounds": int(r.size)}


def variant_summary(c, w, chunk, world, pk):
    """A one-byte-code layer: prefill chunk against the tensor peak, its two
    GEMMs, and batch-1 decode against HBM."""
    fl = {n: gemm_flops(c, chunk, n) for n in ("gate_up", "down")}
    tf = (fl["gate_up"] + fl["down"]) / w["t_pre"] / 1e12
    b = decode_bytes(c, 1, bits=w["bits"])
    gk = {n: w["k_pre"].get(f"gemm_{n}") for n in fl}
    return {"layer": f"same shape as the step's layer, {w['bits']}-bit codes, {W8_REPLICAS} distinct layers for decode",
            "prefill": {"ms_per_4096_chunk": 1e3 * w["t_pre"], "tok_s": job_value(chunk, world, w["t_pre"]),
                        "tensor_tflops": tf, "frac_of_burst_peak": tf / pk["bf16_tflops"],
                        "frac_of_sustained_peak": tf / pk["bf16_tflops_sustained"],
                        "gemm_us": {n: 1e6 * t for n, t in gk.items() if t},
                        "gemm_frac_of_burst_peak": {n: fl[n] / t / 1e12 / pk["bf16_tflops"]
                                                    for n, t in gk.items() if t}},
            "decode_T1": {"us_per_call": 1e6 * w["t_dec"], "bytes_per_call": b, "hbm_gbs": b / w["t_dec"] / 1e9,
                          "frac_of_hbm": b / w["t_dec"] / 1e9 / pk["hbm_gbs"],
                          "path": "one-kernel batch-1 decode (decode_fused_kernel, one-byte-code instance)"}}


# ---------------------------------------------------------------------------
# CPU oracle (baseline arm and the cpu_baseline object)
# ---------------------------------------------------------------------------
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def time_oracle(L0, x_np, n_prefill, n_decode, xdec_np):
    import oracle as O
    t0 = time.perf_counter()
    O.moe_layer(L0, x_np[:n_prefill])
    for i in range(n_decode):
        O.moe_layer(L0, xdec_np[i:i + 1])
    dt = time.perf_counter() - t0
    return (n_prefill + n_decode) / dt, dt


def run_reference(args):
    """The oracle as it stands, on this host's cores: each step is a bounded
    sample of the workload (8 prefill rows and one decode row)."""
    from bit_quantized_sparse_gb300 import synthetic as S
    c = S.CONFIGS[WORKLOAD]
    L0, x = S.draw_config(WORKLOAD, T=64)
    xdec = S.draw_tokens(L0, 4, c["seed"], stream=1)
    for _ in range(args.warmup):
        time_oracle(L0, x, 8, 1, xdec)
    times = [time_oracle(L0, x, 8, 1, xdec)[1] for _ in range(args.steps)]
    total = sum(times)
    val = 9 * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: H=2048 E=256 top-8 I=512 Zipf(1.2); step = 8 prefill rows + 1 decode row"},
            "cpu_baseline": {"value": val, "unit": "tok/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": "8 prefill rows + 1 decode row per step of the long_T16384 layer"},
            "e2e": {"value": val, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.case != "step":
        run_case(args)
        return
    import torch
    dist = init_dist(world, "nccl")
    r = run_gpu(args, rank, local_rank, world, dist)
    c = r["c"]
    pk = peaks()
    T, ndec, chunk = c["T"], c["decode_steps"], c["chunk"]
    units = T + ndec
    value = job_value(units, world, r["t_step"] / args.steps)
    pre_tok_s = job_value(T, world, r["t_pre"] / args.steps)
    dec_tok_s = job_value(ndec, world, r["t_dec"] / args.steps)

    # dominant kernel of the step: largest total time share (4 prefill calls + 64 decode calls)
    share = {("prefill", n): 4 * t for n, t in r["k_pre"].items()}
    share.update({("decode", n): ndec * t for n, t in r["k_dec"].items()})
    total = sum(share.values())
    dom = max(share, key=share.get)
    t_dom = r["k_pre" if dom[0] == "prefill" else "k_dec"][dom[1]]
    if dom[1] in ("gemm_gate_up", "gemm_down"):
        f = gemm_flops(c, chunk, "gate_up" if dom[1] == "gemm_gate_up" else "down")
        ach = f / t_dom / 1e12
        gk = "grouped_w4_gemm_kernel<1, 4, 0>" if dom[1] == "gemm_gate_up" else "grouped_w4_gemm_kernel<0, 4, 0>"
        roof = {"kernel": dom[1], "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "traffic": measured_traffic(gk),
                "work_per_launch": f"{f:.4e} FLOP (fp16 operands, fp32 accumulate)",
                "peak_note": f"dense bf16 burst (the kernel is timed in short replays), {pk['source']}; fp16 has "
                             f"the same nominal rate"}
    else:
        b = decode_bytes(c)
        fused_only = len(r["k_dec"]) == 1
        # one fused launch per call: the decode region of the step is 64 consecutive
        # launches of this kernel alone, so its average launch duration is that
        # region's CUDA-event time over the launches (back to back, as in the step;
        # the traced duration of a launch isolated between events is reported too)
        t_launch = r["t_dec"] / args.steps / ndec if fused_only else sum(r["k_dec"].values())
        ach = b / t_launch / 1e9
        roof = {"kernel": "decode_fused_kernel" if fused_only else "decode step", "bound": "hbm", "achieved": ach,
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
                "traffic": measured_traffic("decode_fused_kernel") if fused_only else None,
                "work_per_launch": f"{b} B (algorithmic bytes of one batch-1 call)",
                "us_per_launch": 1e6 * t_launch,
                "duration": ("decode region of the timed replays: CUDA events around 64 consecutive launches, "
                             "averaged" if fused_only else "sum of the traced kernels of one call"),
                "us_isolated_launch": 1e6 * sum(r["k_dec"].values()),
                "peak_note": f"measured copy bandwidth, {pk['source']}"}
    fused = len(r["k_dec"]) == 1
    t_dec_call = r["t_dec"] / args.steps / ndec if fused else sum(r["k_dec"].values())
    dec_launches = len(r["k_dec"])
    dec_b = decode_bytes(c)
    roof_dec = {"kernel": "decode_fused_kernel" if fused else "decode call (3 kernels)", "bound": "hbm", "achieved": dec_b / t_dec_call / 1e9,
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": dec_b / t_dec_call / 1e9 / pk["hbm_gbs"],
                "bytes_per_call": dec_b, "us_per_call": 1e6 * t_dec_call,
                "us_isolated_launch": 1e6 * sum(r["k_dec"].values()),
                "traffic": measured_traffic("decode_fused_kernel") if fused else None,
                "us_per_call_in_step": 1e6 * r["t_dec"] / args.steps / ndec}
    pre_flops = gemm_flops(c, chunk, "gate_up") + gemm_flops(c, chunk, "down")
    t_chunk = r["t_pre"] / args.steps / (T // chunk)
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * r["t_step"] / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16-mma/fp32-acc (w4 codes, bf16 in/out)",
            "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: T=16384 prefill in 4x4096 chunks + 64 decode steps; H=2048 E=256 "
                                   f"top-8 I=512 shared expert, Zipf(1.2) routing",
                       "l2": f"inputs larger than L2: 455 MB of weights per layer; decode cycles {N_REPLICAS} "
                             f"distinct layers ({N_REPLICAS * 455} MB)",
                       "parallelism": f"replicas x{world}",
                       "timing": "CUDA graph replay, CUDA events around every replay on the replay stream; "
                                 "clocks sampled every 20 ms across all timed regions"},
            "prefill": {"tok_s": pre_tok_s, "ms_per_4096_chunk": 1e3 * t_chunk,
                        "tensor_tflops": pre_flops / t_chunk / 1e12,
                        "frac_of_burst_peak": pre_flops / t_chunk / 1e12 / pk["bf16_tflops"],
                        "frac_of_sustained_peak": pre_flops / t_chunk / 1e12 / pk["bf16_tflops_sustained"],
                        "gemm_frac_of_burst_peak": {
                            n: gemm_flops(c, chunk, n) / r["k_pre"][f"gemm_{n}"] / 1e12 / pk["bf16_tflops"]
                            for n in ("gate_up", "down") if r["k_pre"].get(f"gemm_{n}")},
                        "ms_per_4096_chunk_spread": spread(r["per_pre"], 1e3 / (T // chunk))},
            "decode": {"tok_s": dec_tok_s, "us_per_token": 1e6 * r["t_dec"] / args.steps / ndec,
                       "us_per_token_spread": spread(r["per_dec"], 1e6 / ndec),
                       "roofline": roof_dec},
            "ms_per_step_spread": spread(r["per_step"], 1e3),
            "decode_multirow": {f"T{Tm}": {"us_per_call": 1e6 * t, "tok_s": job_value(Tm, world, t),
                                           "distinct_experts_per_call": dx,
                                           "bytes_per_call": decode_bytes_rows(c, Tm, dx),
                                           "hbm_gbs": decode_bytes_rows(c, Tm, dx) / t / 1e9,
                                           "frac_of_hbm": decode_bytes_rows(c, Tm, dx) / t / 1e9 / pk["hbm_gbs"],
                                           "path": MULTIROW_PATHS[p],
                                           "other_path_us_per_call": None if ta is None else 1e6 * ta}
                                for Tm, (t, dx, p, ta) in r["small"].items()},
            "format_variants": {v: variant_summary(c, w, chunk, world, pk) for v, w in r["variants"].items()},
            "roofline": roof,
            "kernels_us": {"prefill_4096": {k: 1e6 * v for k, v in r["k_pre"].items()},
                           "decode_T1": {k: 1e6 * v for k, v in r["k_dec"].items()},
                           **({"decode_T4": {k: 1e6 * v for k, v in r["k_dec4"].items()}} if r["k_dec4"] else {})},
            "kernel_share": {f"{a}:{b}": v / total for (a, b), v in sorted(share.items(), key=lambda kv: -kv[1])},
            "gpu_launches": args.steps * (4 * len(PREFILL_KERNELS) + ndec * dec_launches),
            "decode_path": "one fused kernel (decode_fused_kernel)" if fused else "three kernels",
            "e2e": {"value": job_value(units, world, r["t_e2e"] / args.steps), "unit": "tok/s",
                    "h2d_bytes_per_step": units * c["H"] * 2, "d2h_bytes_per_step": units * c["H"] * 2},
            "clocks": r["clocks"], "gpu": r["gpu"],
            **({"ablations": r["ablations"]} if r.get("ablations") else {}),
            "context": {"pages_whole_model_M5_Max": {"prefill_tok_s_4K": 5749.9, "decode_tok_s_4K": 186.6,
                                                    "mlx_lm_prefill": 4737.5, "mlx_lm_decode": 140.9,
                                                    "note": "whole 40-layer model on an Apple M5 Max; context only"}}}
    if rank == 0 and not args.no_cpu_baseline:
        n_pre, n_dec = CPU_SAMPLE
        val, dt = time_oracle(r["L0"], r["x_np"], n_pre, n_dec, r["xdec_np"])
        line["cpu_baseline"] = {"value": val, "unit": "tok/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": f"{n_pre} prefill rows (two 4096-row chunks) + {n_dec} batch-1 decode rows "
                                          f"of the workload ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
