"""Benchmark of the MXFP4 routed-expert MoE layer on GB300.

Default workload: one Kimi-K3-shaped MoE layer at decode batch 1 (hidden
7168, 896 MXFP4 experts of 17,547,264 B resident in HBM, top-16, two bf16
shared experts), synthetic weights and tokens. A step is one forward of the
whole layer (router, top-k, 16 experts, shared experts, combine) for a fresh
token. L2 is flushed (a 256 MiB write) before every timed step, outside the
timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 1|2|3|4] [--tokens T] [--graph]
                  [--cache-slots N [--token-corr RHO]] [--no-cpu-baseline]

Prints one JSON line on rank 0. Under torchrun (N > 1) every rank runs an
independent replica on its own GPU (the layer does not shard: replicas only);
time is the max over ranks and the value sums the tokens of all ranks.
--impl reference times the CPU oracle (the plain reference implementation) on
the host cores on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "K3-shape MoE-layer decode tokens/s; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
TOKEN_POOL = 64
REF_TIMED_SECONDS = 120  # cap on the reference arm's timed oracle tokens


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", type=int, default=1, choices=[1, 2, 3, 4])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--tokens", type=int, default=0,
                   help="override the tokens per step of the workload (the stack "
                        "workload decodes at batch 1 and batch 4)")
    p.add_argument("--graph", action="store_true",
                   help="replay the forward pass as one CUDA graph (df_moe_graph_*); each "
                        "step's token is copied into the graph's input buffer before the "
                        "step's timed region, with the L2 flush")
    p.add_argument("--mma-sync-prefill", action="store_true",
                   help="batches above 8 tokens on the register-fragment expert kernels "
                        "instead of the tcgen05 GEMMs (DF_MOE_PREFILL_MMA_SYNC)")
    p.add_argument("--cache-slots", type=int, default=0,
                   help="experts in pinned host memory, this many a layer cached in HBM "
                        "(df_moe_create_cached); decode batches only")
    p.add_argument("--token-corr", type=float, default=0.0,
                   help="consecutive steps take consecutive tokens of a stream whose "
                        "neighbours have this correlation (0.7: ~31%% of the experts "
                        "reused from the previous token); 0: independent tokens")
    p.add_argument("--mxfp8", action="store_true",
                   help="the lossy MXFP8-activation variant (DF_MOE_MXFP8_ACT): routed "
                        "experts on block-scaled MXFP4 x MXFP8 tcgen05 GEMMs")
    p.add_argument("--planes", action="store_true",
                   help="exact batches on the block-scaled MXFP4 x E4M3 tcgen05 GEMMs, "
                        "activations as sums of E4M3 planes (DF_MOE_PLANES); the default "
                        "for batch workloads (more than 8 tokens a step)")
    p.add_argument("--no-planes", action="store_true",
                   help="4 tokens or more on a default handle (the decode kernels up to 8 "
                        "tokens, the GEMMs with MXFP4 decoded into tensor memory above) "
                        "instead of the planes")
    p.add_argument("--experts", type=int, default=0,
                   help="profiling aid: override the routed-expert count (same "
                        "per-token work, smaller resident set); not a bench line")
    return p.parse_args()


# ---- byte accounting ----------------------------------------------------------

def layer_bytes(wl, n_union, T):
    """Algorithmic HBM bytes of one layer call: router + shared experts + every
    distinct selected expert read once + x in and out (bf16)."""
    span = synth.span_bytes(wl.H, wl.I)
    router = wl.E * wl.H * 4
    shared = wl.n_shared * 3 * wl.Is * wl.H * 2
    return router + shared + n_union * span + T * wl.H * 2 * 2


def gateup_bytes(wl, n_union, T, with_shared=False):
    """Algorithmic bytes of the gate/up kernel: the gate and up halves of every
    distinct selected expert (codes + scales), x in, h out (fp32); with_shared:
    also the shared experts' gate and up rows (bf16) and their h (the decode
    phase kernel runs both)."""
    per_expert = 2 * wl.I * wl.H * 17 // 32
    b = n_union * per_expert + T * wl.H * 2 + T * wl.k * wl.I * 4
    if with_shared:
        b += wl.n_shared * 2 * wl.Is * wl.H * 2 + T * wl.n_shared * wl.Is * 4
    return b


def mx8_gateup_bytes(wl, n_union, T, planes=1):
    """Algorithmic bytes of the block-scaled gate/up GEMM: the gate and up
    halves of every distinct selected expert (codes + scales) and the E4M3 x
    rows of the T*k assignments (`planes` rows each) with their scales in;
    out, the E4M3 h rows with their scales (MXFP8) or h in fp32 (planes)."""
    per_expert = 2 * wl.I * wl.H * 17 // 32
    rows = T * wl.k
    h_out = rows * (wl.I + wl.I // 32) if planes == 1 else rows * wl.I * 4
    return n_union * per_expert + rows * planes * (wl.H + wl.H // 32) + h_out


def mx8_phase_gateup_bytes(wl, n_union):
    """Algorithmic bytes of the one-token gate/up phase kernel of an exact-planes
    handle: the routed experts' gate and up halves (codes + scales) and x's four
    E4M3 planes in, the gate and up sums of its eight parts of K out (fp32),
    and beside them the shared experts' gate and up rows (bf16), x (bf16) and
    their h (fp32)."""
    per_expert = 2 * wl.I * wl.H * 17 // 32
    kspl = max(1, min(8, wl.H // 128))
    routed = n_union * per_expert + 4 * (wl.H + wl.H // 32) + kspl * wl.k * 2 * wl.I * 4
    shared = wl.n_shared * 2 * wl.Is * wl.H * 2 + wl.H * 2 + wl.n_shared * wl.Is * 4
    return routed + shared


def gateup_flops(wl, T):
    """Useful flops of the routed gate/up contraction: 2 per multiply-add of
    each of the T*k assignments' 2I x H products."""
    return 2.0 * T * wl.k * 2 * wl.I * wl.H


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


# The sources each recorded kernel's DRAM traffic depends on: a change to any
# of them voids the record.
KERNEL_SOURCES = {
    "expert_gateup": ("k_phase.cu", "mxv.cuh", "bfv.cuh", "select.cuh", "mxfrag.cuh",
                      "pipeline.cuh"),
    "expert_down": ("k_phase.cu", "mxv.cuh", "bfv.cuh", "mxfrag.cuh", "pipeline.cuh"),
    "gemm_gateup": ("k_gemm.cu", "umma.cuh", "mxfrag.cuh", "pipeline.cuh"),
    "gemm_down": ("k_gemm.cu", "umma.cuh", "mxfrag.cuh", "pipeline.cuh"),
    "mx8_gateup": ("k_mx8.cu", "umma.cuh", "pipeline.cuh", "bfv.cuh", "select.cuh"),
    "mx8_down": ("k_mx8.cu", "umma.cuh", "pipeline.cuh", "bfv.cuh", "select.cuh"),
}


def csrc_hash(kernel=None):
    """Hash of the CUDA sources a kernel kind's traffic depends on (all of
    csrc/ for an unknown kind)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mxfp4_routed_expert_top_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(
        n for n in os.listdir(d) if n.endswith((".cu", ".h", ".cuh")))
    for name in sorted(names):
        h.update(name.encode())
        h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, wl, planes=0):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the
    kernel's sources have not changed since it was captured and a launch of
    workload `wl` does the captured launch's work (same tokens a layer and
    experts); else None. The exact-planes GEMMs are recorded apart (their
    activation rows are several times larger)."""
    try:
        d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        rec = d.get(kernel + ("_planes" if planes else ""))
        if (rec and rec.get("csrc_hash") == csrc_hash(kernel) and rec.get("tokens") == wl.T
                and rec.get("experts") == wl.E and rec.get("hidden") == wl.H):
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ---- clocks -----------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [v.strip() for v in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


# ---- distributed --------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate_over_ranks(dist, seconds, units, device="cpu"):
    """Max of the elapsed time and sum of the units over ranks (replicas)."""
    import torch
    if dist is None:
        return seconds, units
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---- CPU oracle baseline ------------------------------------------------------

def cpu_oracle_rate(wl, seconds, max_tokens=None):
    """Tokens/s of the CPU oracle on the workload's tokens, timed until
    `seconds` of work (0: no time limit) or `max_tokens` tokens, whichever
    comes first (at least one token). Returns (rate, tokens, threads)."""
    import oracle as orc
    layers = []
    for l in range(wl.L):
        router = synth.router(wl.seed, wl.wcfg, l, wl.E, wl.H)
        shared = [synth.shared(wl.seed, wl.wcfg, l, s, wl.H, wl.Is)
                  for s in range(wl.n_shared)]
        layers.append(orc.Layer(
            wl.H, wl.E, wl.k, wl.I, wl.Is, router, shared,
            lambda ly, e: synth.expert_spans(wl.seed, wl.wcfg, ly, e, 1, wl.H, wl.I)[0],
            layer=l))
    n, t0 = 0, time.perf_counter()
    while True:
        x = synth.token(wl.seed, wl.cfg_id, 100000 + n, wl.H)[None, :]
        if wl.stack:
            orc.moe_stack(layers, x, wl.eps)
        else:
            orc.moe_layer(layers[0], x)
        for L in layers:
            L.clear_cache()
        n += 1
        el = time.perf_counter() - t0
        if (seconds > 0 and el >= seconds) or (max_tokens and n >= max_tokens):
            break
    return n / el, n, orc.num_threads()


# ---- our implementation -------------------------------------------------------

def load_workload(m, wl, torch, stream, chunk=64):
    span = synth.span_bytes(wl.H, wl.I)
    buf = torch.empty(chunk * span, dtype=torch.uint8, device="cuda")
    for l in range(wl.L):
        router = synth.router(wl.seed, wl.wcfg, l, wl.E, wl.H)
        shared = [synth.shared(wl.seed, wl.wcfg, l, s, wl.H, wl.Is)
                  for s in range(wl.n_shared)]
        m.load_experts(l, router=router, shared=shared)
        for e0 in range(0, wl.E, chunk):
            n = min(chunk, wl.E - e0)
            synth.dev_expert_spans(wl.seed, wl.wcfg, l, e0, n, wl.H, wl.I,
                                   buf.data_ptr(), stream.cuda_stream)
            m.load_experts(l, experts=buf, expert_begin=e0, expert_count=n,
                           src_is_device=True, stream=stream)
    torch.cuda.synchronize()
    del buf


def run_ours(args):
    import torch
    import mxfp4_routed_expert_top_gb300 as dfm

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl")
    wl = synth.WORKLOADS[args.config]
    import dataclasses
    if args.experts:
        wl = dataclasses.replace(wl, E=args.experts, name=wl.name + "-e%d" % args.experts)
    if args.tokens:
        wl = dataclasses.replace(wl, T=args.tokens, name=wl.name + "-t%d" % args.tokens)
    T = wl.T
    # from 4 tokens on, layers run on the exact planes (the faster exact path
    # there: 326 against 331 us at 4 tokens, 487 against 606 at 8) unless
    # another path is asked for; fewer tokens run on the decode kernels
    if (T >= 4 and not (args.no_planes or args.mxfp8 or args.mma_sync_prefill or args.cache_slots
                        or wl.stack)):
        args.planes = True
    flags = ((dfm.STACK_RMSNORM_RESIDUAL if wl.stack else 0)
             | (dfm.PREFILL_MMA_SYNC if args.mma_sync_prefill else 0)
             | (dfm.MXFP8_ACT if args.mxfp8 else 0)
             | (dfm.PLANES if args.planes else 0))
    if args.cache_slots and T > 8:
        raise SystemExit("--cache-slots serves decode batches (<= 8 tokens)")
    m = dfm.MoE(wl.H, wl.E, wl.k, wl.I, wl.n_shared, wl.Is, n_layers=wl.L,
                max_tokens=T if args.cache_slots else max(T, 4), rms_eps=wl.eps, flags=flags,
                device=local, cache_slots=args.cache_slots)
    stream = torch.cuda.current_stream()
    load_workload(m, wl, torch, stream)

    # a pool of distinct synthetic tokens (fresh x each step), resident in HBM;
    # a correlated stream runs through the warm-up and the timed steps
    # without wrapping
    n_pool = TOKEN_POOL
    if args.token_corr:
        n_pool = max(TOKEN_POOL, args.warmup + args.steps)
        pool = synth.token_stream(wl.seed, wl.cfg_id, 0, n_pool * T, wl.H, args.token_corr,
                                  stream=1 + rank).reshape(n_pool, T, wl.H)
    else:
        pool = np.stack([synth.token(wl.seed, wl.cfg_id, 200000 + rank * 100000 + i, wl.H)
                         for i in range(n_pool * T)]).reshape(n_pool, T, wl.H)
    xs = torch.from_numpy(pool.view(np.int16)).cuda()
    out = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
    ids = torch.empty((wl.L, T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.L, T, wl.k), dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    graph = None
    if args.graph:
        x_cur = xs[0].clone()
        graph = m.graph(x_cur, T, out, ids, w)

        def stage(i):  # outside the timed region, beside the flush
            x_cur.copy_(xs[i % n_pool])

        def step(i):
            graph.launch(stream=stream)
    else:
        def stage(i):
            pass

        def step(i):
            m.forward(xs[i % n_pool], T, out, ids, w, stream=stream)

    def launches_of_step():
        return graph.launch_count() if graph is not None else m.last_launch_count()

    for i in range(args.warmup):
        stage(i)
        flush.fill_(float(i))
        step(i)
    m.sync(stream)

    # timed region: K steps, per-step CUDA events around the forward only
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    n_union = []
    launches = 0
    with ClockSampler(local) as clk:
        barrier(dist)
        torch.cuda.synchronize()
        # The sampler's start leaves the GPU idle for a third of a second, and
        # the first step after such an idle spell ran ~24 us long at batch 1
        # (the slowest step of every run). Two untimed steps (the warm-up's
        # last tokens again), queued straight ahead of the timed ones, bring
        # the GPU back and give the host a head start, as every later step has.
        for j in range(2):
            i = max(args.warmup - 2 + j, 0)
            stage(i)
            flush.fill_(float(i))
            step(i)
        cache0 = m.cache_stats()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            stage(i)
            flush.fill_(float(i))
            starts[i].record(stream)
            step(i)
            ends[i].record(stream)
            launches += launches_of_step()
        torch.cuda.synchronize()
        barrier(dist)
        wall = time.perf_counter() - wall0
    m.sync(stream)
    cache1 = m.cache_stats()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dev_s = sum(step_ms) / 1e3
    # distinct experts per step (for the byte count), from the ids of the
    # pool; and the share of a step's experts that the step before selected
    prev, reuse = None, []
    for i in range(min(args.steps, n_pool)):
        m.forward(xs[i], T, out, ids, w, stream=stream)
        sel = set(np.unique(ids[0].cpu().numpy()).tolist())
        n_union.append(len(sel))
        if prev is not None:
            reuse.append(len(sel & prev) / len(sel))
        prev = sel
    u_mean = float(np.mean(n_union))

    # per-kernel device time (same steps, library events on the same stream)
    m.timing_reset()
    m.timing_enable(True)
    for i in range(min(args.steps, 50)):
        flush.fill_(float(i))
        m.forward(xs[i % n_pool], T, out, ids, w, stream=stream)
    kt = m.timing()
    m.timing_enable(False)

    # the read-only streaming rate of this GPU (our probe kernel over 1 GiB)
    probe = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    sink = torch.empty(8 * torch.cuda.get_device_properties(local).multi_processor_count * 256,
                       dtype=torch.int32, device="cuda")
    probe_ms = []
    for i in range(8):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dfm.stream_read(probe, probe.numel(), sink, stream=stream)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            probe_ms.append(a.elapsed_time(b))
    stream_read_gbs = probe.numel() / (float(np.median(probe_ms)) / 1e3) / 1e9
    del probe, sink

    cache = None
    if args.cache_slots:
        # the ceiling of the cache's copies: pinned host -> HBM copy rate, as
        # one 1 GiB copy and as 16 expert-span copies (one token's misses)
        span = m.span_bytes
        hsrc = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
        ddst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")

        def h2d_gbs(nbytes, pieces):
            t = []
            for i in range(6):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for j in range(pieces):
                    ddst[j * nbytes:(j + 1) * nbytes].copy_(hsrc[j * nbytes:(j + 1) * nbytes],
                                                           non_blocking=True)
                b.record(stream)
                b.synchronize()
                if i >= 2:
                    t.append(a.elapsed_time(b))
            return nbytes * pieces / (float(np.median(t)) / 1e3) / 1e9

        copy_gbs, burst_gbs = h2d_gbs(1 << 30, 1), h2d_gbs(span, 16)
        del hsrc, ddst
        dh, dm, db = (cache1[i] - cache0[i] for i in range(3))
        ntok = T * args.steps
        cache = {"slots_per_layer": args.cache_slots, "hits": dh, "misses": dm,
                 "hit_rate": round(dh / max(dh + dm, 1), 4),
                 "bytes_in_per_token": int(round(db / ntok)),
                 "bytes_in_gbs": round(db / dev_s / 1e9, 1),
                 "h2d_copy_gbs": round(copy_gbs, 1),
                 "h2d_16_span_copies_gbs": round(burst_gbs, 1),
                 "frac_of_h2d_copy": round(db / dev_s / 1e9 / copy_gbs, 4),
                 "reuse_of_previous_step": round(float(np.mean(reuse)), 4) if reuse else None}

    # end to end through the public API with host buffers (pinned)
    hx = torch.from_numpy(pool.view(np.int16)).pin_memory()
    hout = torch.empty((T, wl.H), dtype=torch.int16).pin_memory()
    hids = torch.empty((wl.L, T, wl.k), dtype=torch.int32).pin_memory()
    hw = torch.empty((wl.L, T, wl.k), dtype=torch.float32).pin_memory()
    e2e_steps = min(args.steps, 50)
    e2e_t = []
    for i in range(e2e_steps + 3):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        m.forward_host(hx[i % n_pool], T, hout, ids=hids, weights=hw, stream=stream)
        if i >= 3:
            e2e_t.append(time.perf_counter() - t0)
    e2e_s = sum(e2e_t)
    # where the host-buffer call's time goes. The call moves its data on the
    # device (a copy kernel pulls x from pinned host memory, the last kernel
    # writes out, ids and weights into it); for scale, the same bytes as DMA
    # copies on their own (each followed by a synchronisation) and an empty
    # synchronisation
    xdev = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")

    def host_us(fn, n=50):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        return (time.perf_counter() - t0) / n * 1e6

    def h2d():
        xdev.copy_(hx[0], non_blocking=True)
        stream.synchronize()

    def d2h():
        hout.copy_(out, non_blocking=True)
        hids.copy_(ids, non_blocking=True)
        hw.copy_(w, non_blocking=True)
        stream.synchronize()

    call_us = e2e_s / max(len(e2e_t), 1) * 1e6
    h2d_us, d2h_us, sync_us = host_us(h2d), host_us(d2h), host_us(stream.synchronize)
    dev_us = float(np.median(step_ms)) * 1e3
    e2e_breakdown = {"call_us": round(call_us, 1), "device_step_us": round(dev_us, 1),
                     "call_minus_device_step_us": round(call_us - dev_us, 1),
                     "in_call_transfers": "device-side: copy kernel in, last kernel writes out",
                     "dma_h2d_copy_and_sync_us": round(h2d_us, 1),
                     "dma_d2h_copies_and_sync_us": round(d2h_us, 1),
                     "empty_sync_us": round(sync_us, 1)}

    dev_s_max, tokens = aggregate_over_ranks(dist, dev_s, T * args.steps, device="cuda")
    e2e_max, e2e_tokens = aggregate_over_ranks(dist, e2e_s, T * e2e_steps, device="cuda")
    if rank != 0:
        if graph is not None:
            graph.close()
        m.close()
        return None

    peak, peak_kind = measured_peaks()
    ms = dev_s_max / args.steps * 1e3
    lb = layer_bytes(wl, u_mean, T) * wl.L
    # dominant kernel: the routed gate/up GEMM (tcgen05, larger batches),
    # else the gate/up phase of decode batches
    if kt.get("mx8_gateup", (0, 0.0))[0] and args.planes and T == 1 and not args.cache_slots:
        # one token on exact planes: the gate/up phase kernel, shared experts
        # beside the routed ones
        dom, dom_bytes = "mx8_gateup", mx8_phase_gateup_bytes(wl, u_mean)
    elif kt.get("mx8_gateup", (0, 0.0))[0]:
        dom, dom_bytes = "mx8_gateup", mx8_gateup_bytes(wl, u_mean, T, 4 if args.planes else 1)
    elif kt.get("gemm_gateup", (0, 0.0))[0]:
        dom, dom_bytes = "gemm_gateup", gateup_bytes(wl, u_mean, T)
    else:
        # decode batches: the gate/up phase kernel streams the routed and the
        # shared experts' gate/up rows
        dom, dom_bytes = "expert_gateup", gateup_bytes(wl, u_mean, T, with_shared=T <= 8)
    dom_n, dom_ms = kt[dom]
    dom_avg_ms = dom_ms / max(dom_n, 1)
    dom_gbs = dom_bytes / (dom_avg_ms / 1e3) / 1e9
    layer_gbs = lb / (ms / 1e3) / 1e9
    kernels = {k: {"launches": n, "avg_us": round(t / max(n, 1) * 1e3, 2)}
               for k, (n, t) in kt.items() if n}
    res = {
        "metric": METRIC, "value": round(tokens / dev_s_max, 2), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e2m1 x e4m3, f32 accumulate" if args.mxfp8 else
                  "e2m1 x e4m3 planes, f32 accumulate" if args.planes else "f32"),
        "data": "synthetic",
        "impl": "ours",
        "config": {**workload_config(wl, ws),
                   "l2": "flushed (256 MiB write) before every timed step",
                   "launch": "cuda graph" if args.graph else "stream",
                   "expert_path": ("decode phase kernels with the routed experts on the tcgen05 "
                                   "block-scaled MMA (E4M3 planes) beside the shared GEMV"
                                   if args.planes and T == 1 and not args.cache_slots else
                                   "tcgen05 block-scaled (E4M3 planes)" if args.planes else
                                   "tcgen05 block-scaled (MXFP8)" if args.mxfp8 else
                                   "decode phase kernels (mma.sync GEMVs)" if T <= 8 else
                                   "mma_sync" if args.mma_sync_prefill else
                                   "tcgen05 (MXFP4 decoded into tensor memory)"),
                   "activations": ("MXFP8 (E4M3, E8M0 per 32) into the routed experts: "
                                   "the lossy variant") if args.mxfp8 else
                                  ("exact, as sums of E4M3 planes (x 4, h 5) on the "
                                   "block-scaled GEMMs") if args.planes else "exact",
                   "experts_home": ("pinned host memory, %d a layer cached in HBM"
                                    % args.cache_slots) if args.cache_slots else "HBM",
                   "tokens": ("AR(1) stream, neighbour correlation %g" % args.token_corr)
                             if args.token_corr else "independent N(0,1)"},
        "step_us": {"median": round(float(np.median(step_ms)) * 1e3, 2),
                    "mean": round(float(np.mean(step_ms)) * 1e3, 2),
                    "p10": round(float(np.percentile(step_ms, 10)) * 1e3, 2),
                    "p90": round(float(np.percentile(step_ms, 90)) * 1e3, 2),
                    "max": round(float(np.max(step_ms)) * 1e3, 2),
                    "max_step": int(np.argmax(step_ms))},
        "layer_hbm": {"achieved_gbs": round(layer_gbs, 1), "bytes_per_step": int(lb),
                      "frac_of_measured": round(layer_gbs / peak, 4),
                      "stream_read_gbs": round(stream_read_gbs, 1),
                      "frac_of_stream_read": round(layer_gbs / stream_read_gbs, 4),
                      "frac_of_nominal_8tbs": round(layer_gbs / 8000.0, 4),
                      "distinct_experts_per_step": u_mean},
        "roofline": {"bound": "hbm", "kernel": dom,
                     "achieved": round(dom_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dom_gbs / peak, 4), "peak_source": peak_kind,
                     "bytes_per_launch": int(dom_bytes),
                     "traffic": recorded_traffic(dom, wl, 4 if args.planes else 0)},
        "kernels": kernels,
        "tensor": tensor_use(kt, wl, T),
        "e2e": {"value": round(e2e_tokens / e2e_max, 2), "unit": UNIT,
                "h2d_bytes_per_step": T * wl.H * 2,
                "d2h_bytes_per_step": T * wl.H * 2 + wl.L * T * wl.k * 8,
                "breakdown": e2e_breakdown},
        "gpu_launches": launches,
        **({"cache": cache} if cache else {}),
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    if graph is not None:
        graph.close()
    m.close()
    return res


def tensor_use(kt, wl, T):
    """Useful bf16 tensor throughput of the gate/up GEMM (tcgen05 path only):
    the assignments' flops over its average launch time, against the
    measured dense bf16 peak. At a few tokens per expert the GEMM is HBM
    bound, so this fraction is small by construction."""
    kern, ratio = "gemm_gateup", 1.0
    n, t = kt.get(kern, (0, 0.0))
    if not n:
        # the MXFP8 variant: E4M3 x E2M1 on the fp8 pipe, nominally twice bf16
        kern, ratio = "mx8_gateup", 2.0
        n, t = kt.get(kern, (0, 0.0))
    if not n:
        return None
    peak, src = measured_bf16_tflops()
    peak *= ratio
    if ratio != 1.0:
        src += " bf16 x 2 (nominal fp8/bf16 ratio)"
    tf = gateup_flops(wl, T) / (t / n / 1e3) / 1e12
    return {"kernel": kern, "achieved": round(tf, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(tf / peak, 4), "peak_source": src}


def workload_config(wl, ws):
    """The workload keys of the JSON line's config, shared by both arms."""
    return {"workload": wl.name, "hidden": wl.H, "experts": wl.E, "top_k": wl.k,
            "inter": wl.I, "shared": wl.n_shared, "tokens_per_step": wl.T,
            "layers": wl.L, "weights": "mxfp4 e2m1+e8m0/32, shared bf16",
            "parallelism": "replicas" if ws > 1 else "single-gpu"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return None
    wl = synth.WORKLOADS[args.config]
    if args.tokens:
        import dataclasses
        wl = dataclasses.replace(wl, T=args.tokens, name=wl.name + "-t%d" % args.tokens)
    # each step: one token of the workload through the oracle (a bounded
    # sample of the workload: the oracle is per-token, so tokens/s carries over)
    # at most a minute of warm-up and two of timed tokens, so that the whole
    # run ends within minutes at every workload
    cpu_oracle_rate(wl, 60.0, max_tokens=max(args.warmup, 1))
    t0 = time.perf_counter()
    rate, n, threads = cpu_oracle_rate(wl, REF_TIMED_SECONDS, max_tokens=args.steps)
    el = time.perf_counter() - t0
    value = n / el
    return {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / n * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(wl, ws),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": "%d tokens of %s (%d of %d steps within the %d s cap), one "
                                   "token through the oracle per step (its cost is per token)"
                                   % (n, wl.name, n, args.steps, REF_TIMED_SECONDS)},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_ours(args)
        if res is not None and not args.no_cpu_baseline:
            wl = synth.WORKLOADS[args.config]
            rate, n, threads = cpu_oracle_rate(wl, args.cpu_seconds)
            res["cpu_baseline"] = {
                "value": round(rate, 4), "unit": UNIT,
                "cores": threads, "kind": "oracle",
                "sample": "%d tokens of %s through the CPU oracle (%.1f s)" % (
                    n, wl.name, n / rate)}
            # the same oracle on one core (a third of the time budget)
            import oracle as orc
            orc.set_num_threads(1)
            try:
                r1, n1, _ = cpu_oracle_rate(wl, args.cpu_seconds / 3)
            finally:
                orc.set_num_threads(threads)
            res["cpu_baseline"]["single_thread"] = {
                "value": round(r1, 4), "unit": UNIT, "cores": 1,
                "sample": "%d tokens, %.1f s" % (n1, n1 / r1)}
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
