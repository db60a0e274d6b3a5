"""Benchmark of the MoE layer hot path on GB300: one step = one pass of the whole layer
(route -> permute -> grouped GEMM gate/up + SwiGLU -> grouped GEMM down -> combine)
over one batch of the prefill workload (T = 8192 tokens in a 16384-row bucket,
H = 7168, I = 2048, E = 256, top-8, one shared expert, BF16, Zipf(1.1) router skew).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--layout contiguous|batched [--max-tokens M]] [--fuse-combine]

Prints one JSON line (rank 0).  `value` is layer tokens/s with inputs resident in HBM;
`e2e` is the same metric through moe_layer_forward with the step's inputs copied from
pinned host memory and its output copied back inside the timed region.  The per-kernel
breakdown (and the roofline of the dominant kernel) comes from a second timed pass that
issues the same steps through the per-step C calls with CUDA events between them.
Inputs are synthetic (seeded); the weights (22.6 GB) are far larger than L2, so every
step streams them from HBM without an explicit flush.

`--impl reference` times the CPU oracle (plain numpy, as it stands) on a bounded sample
of the same workload on the host cores.  With --gpus N > 1 the script starts N ranks of
one node itself (torch.distributed.run on 127.0.0.1) unless torchrun already did; each
rank runs an independent batch on its own GPU (token-sharded replicas, no collective in
the data path), timing is the max over ranks and rank 0 prints the line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from combine_moe_route_softmax_gb300 import synth  # noqa: E402

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ distributed glue
def dist_env():
    """(rank, world, local_rank) from torchrun's environment (1-process defaults)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value, world, device="cpu"):
    """Largest value over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed, rank):
    """Each rank draws its own batch (weak scaling); the weights are shared (same seed)."""
    return seed + 1000 * rank


def max_stage_times(stage_ms, world, device="cpu"):
    """Per-stage times of this rank -> the slowest rank's time of every stage."""
    return {k: max_over_ranks(v, world, device) for k, v in stage_ms.items()}


def whole_job_rate(units_per_rank, world, ms):
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (ms * 1e-3)


def emit(line, rank):
    """The job's one JSON line, printed by rank 0 only; returns whether this rank printed."""
    if rank != 0:
        return False
    print(json.dumps(line), flush=True)
    return True


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(n, argv):
    """`--gpus N` with N > 1 outside torchrun: run this script again as N ranks of one node
    under torch.distributed.run (rendezvous on 127.0.0.1) and return their exit status;
    None when this process is already a rank (or N == 1) and should do the work itself."""
    if n <= 1 or "WORLD_SIZE" in os.environ:
        return None
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


# ---------------------------------------------------------------------- peaks/clocks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
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
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax = float(p[2])
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------- our arm
def workload_state(w, seed, device, max_tokens=0, fuse_combine=False, dispatch_fq=None, weight_in_down=False,
                   gemm_pairs=False, weight_tiles=False):
    import combine_moe_route_softmax_gb300 as moe
    logits = synth.router_logits(w, seed, device=device)
    x = synth.hidden(w, seed, device=device)
    w13, w2, s13, s2 = synth.expert_weights(w, 0, device=device)   # weights shared by all ranks
    kw = dict(w13=w13, w2=w2, shared_w13=s13, shared_w2=s2)
    dtype = moe.MOE_BF16
    if gemm_pairs and (w.dtype != "bf16" or max_tokens or fuse_combine):
        raise SystemExit("--gemm-pairs applies to BF16 workloads in the contiguous layout without --fuse-combine")
    if w.dtype == "e4m3":
        q13, c13 = moe.moe_quantize_weight_fp8(w13)
        q2, c2 = moe.moe_quantize_weight_fp8(w2)
        kw = dict(w13=q13, w2=q2, w13_scales=c13, w2_scales=c2)
        if w.shared:
            qs13, cs13 = moe.moe_quantize_weight_fp8(s13)
            qs2, cs2 = moe.moe_quantize_weight_fp8(s2)
            kw.update(shared_w13=qs13, shared_w2=qs2, shared_w13_scales=cs13, shared_w2_scales=cs2)
        del w13, w2, s13, s2
        dtype = moe.MOE_E4M3
    layer = moe.MoeLayer(w.T, w.H, w.I, w.E, w.K, dtype, max_tokens=max_tokens, fuse_combine=fuse_combine,
                         weight_in_down=weight_in_down, combine_fq=w.fq_format, dispatch_fq=dispatch_fq or "e4m3",
                         gemm_pairs=gemm_pairs, weight_tiles=weight_tiles, **kw)
    fq = None
    if w.fake_quant:
        # combine fake-quant: the constant scale 448 / amax (E4M3) or the per-tensor scale
        # 448 * 6 / amax (NVFP4), amax calibrated (max) on a batch of 16 tokens drawn with
        # seed + 1 through this layer's own weights (untimed)
        wc = synth.scaled(w, T=16, T_valid=16, fake_quant=False, graph=False)
        cal = moe.MoeLayer(wc.T, wc.H, wc.I, wc.E, wc.K, dtype, **kw)
        c_idx = torch.empty(wc.T, wc.K, dtype=torch.int32, device=device)
        c_wt = torch.empty(wc.T, wc.K, dtype=torch.float32, device=device)
        c_out = torch.empty(wc.T, wc.H, dtype=torch.bfloat16, device=device)
        cal.forward(synth.hidden(wc, seed + 1, device=device), c_out, c_idx, c_wt,
                    logits=synth.router_logits(wc, seed + 1, device=device))
        amax = torch.zeros(1, dtype=torch.float32, device=device)
        cv = cal.views
        moe.moe_combine_amax(cal.view("y", (cv.cap, wc.H), torch.bfloat16),
                             cal.view("inv_map", (wc.T, wc.K), torch.int32), c_wt, amax)
        fq = moe.moe_fq4_scale_from_amax(amax) if w.fq_format == "nvfp4" else moe.moe_fq_scale_from_amax(amax)
        torch.cuda.synchronize()
        del cal
    dq = None
    if dispatch_fq:
        # dispatch fake-quant: the per-tensor scale 448 / max|x| (E4M3) or 448 * 6 / max|x|
        # (NVFP4) over the batch's real tokens (untimed, as a calibration would be)
        if w.dtype != "bf16":
            raise SystemExit("--dispatch-fq applies to BF16 workloads (E4M3 rows are quantised anyway)")
        amax = torch.zeros(1, dtype=torch.float32, device=device)
        moe.moe_amax_bf16(x[:w.T_valid], amax)
        dq = moe.moe_fq4_scale_from_amax(amax) if dispatch_fq == "nvfp4" else moe.moe_fq_scale_from_amax(amax)
        torch.cuda.synchronize()
    # slot padding of the workload (a fixed seeded mask), applied by the harness after routing
    pad = synth.slot_padding(w, seed, device=device) if w.slot_pad > 0 else None
    st = dict(layer=layer, fq=fq, dq=dq, pad=pad, logits=logits, x=x,
              idx=torch.empty(w.T, w.K, dtype=torch.int32, device=device),
              wt=torch.empty(w.T, w.K, dtype=torch.float32, device=device),
              out=torch.empty(w.T, w.H, dtype=torch.bfloat16, device=device),
              n=torch.tensor([w.T_valid], dtype=torch.int32, device=device),
              status=torch.zeros(1, dtype=torch.int32, device=device))
    return st


def layer_step(st, x=None, logits=None, out=None):
    import combine_moe_route_softmax_gb300 as moe
    lg = st["logits"] if logits is None else logits
    if st["pad"] is not None:
        # workloads with padded slots: route, then the harness marks its padding slots -1
        # (weight 0), as a dispatcher would, and the layer runs on those ids
        moe.moe_route_topk(lg, st["idx"].shape[1], num_tokens=st["n"], topk_idx=st["idx"], topk_w=st["wt"])
        st["idx"].masked_fill_(st["pad"], -1)
        st["wt"].masked_fill_(st["pad"], 0.0)
        lg = None
    st["layer"].forward(st["x"] if x is None else x, st["out"] if out is None else out, st["idx"], st["wt"],
                        logits=lg, num_tokens=st["n"], fq_scale=st["fq"], dev_status=st["status"],
                        dispatch_scale=st["dq"])


STAGES = ("route", "permute", "gemm_gate_up", "gemm_down", "combine")


def staged_step(st, w, events):
    """The same step as moe_layer_forward, issued call by call with an event after each."""
    import combine_moe_route_softmax_gb300 as moe
    L = moe.lib()
    lay = st["layer"]
    v, d = lay.views, lay.desc
    s = torch.cuda.current_stream().cuda_stream
    nseg = d.E + d.has_shared
    tw = lay.tensors
    gdt = d.dtype | (moe.MOE_W_TILED if d.weight_tiles else 0)   # the grouped GEMMs' dtype argument
    p = lambda t: None if t is None else t.data_ptr()
    events[0].record()
    assert L.moe_route_topk(p(st["logits"]), d.T, d.E, d.K, p(st["n"]), p(st["idx"]), p(st["wt"]), s) == 0
    if st["pad"] is not None:
        st["idx"].masked_fill_(st["pad"], -1)
        st["wt"].masked_fill_(st["pad"], 0.0)
    events[1].record()
    mt = d.max_tokens
    # router weight in the down projection: the permute emits each row's weight, the down
    # GEMM scales its accumulator by it and the combine only sums
    wd = bool(d.weight_in_down)
    wd_w, wd_rows = (p(st["wt"]), v.row_weights) if wd else (None, None)
    if mt:
        scratch_bytes = L.moe_permute_batched_workspace_bytes(d.T, d.K, d.E, d.has_shared)
    else:
        scratch_bytes = L.moe_permute_workspace_bytes(d.T, d.K, d.E, d.has_shared)
    scratch = st.setdefault("scratch", torch.empty(scratch_bytes, dtype=torch.uint8, device=st["x"].device))
    if mt:
        assert L.moe_permute_batched(p(st["idx"]), d.T, d.K, d.E, d.has_shared, mt, p(st["x"]), d.H, d.dtype, v.xp,
                                     v.xp_scales, v.masked_m, v.src_row, v.inv_map, v.shared_map, p(scratch),
                                     scratch_bytes, p(st["status"]), p(st["dq"]), d.dispatch_fq_format, wd_w,
                                     wd_rows, s) == 0
    elif st["dq"] is not None or wd:
        assert L.moe_permute_ex(p(st["idx"]), d.T, d.K, d.E, d.has_shared, p(st["x"]), d.H, d.dtype, v.xp,
                                v.xp_scales, v.cu_seqlens, v.src_row, v.inv_map, v.shared_map, p(scratch),
                                scratch_bytes, p(st["status"]), p(st["dq"]), d.dispatch_fq_format, wd_w, wd_rows,
                                s) == 0
    else:
        assert L.moe_permute(p(st["idx"]), d.T, d.K, d.E, d.has_shared, p(st["x"]), d.H, d.dtype, v.xp,
                             v.xp_scales, v.cu_seqlens, v.src_row, v.inv_map, v.shared_map, p(scratch),
                             scratch_bytes, p(st["status"]), s) == 0
    events[2].record()
    if mt:
        assert L.moe_grouped_gemm_batched(v.xp, v.xp_scales, v.masked_m, nseg, mt, d.H, 2 * d.I, p(tw[0]), p(tw[4]),
                                          d.E, p(tw[2]), p(tw[6]), gdt, moe.MOE_EPI_SWIGLU, v.hs, v.hs_scales,
                                          p(st["status"]), None, s) == 0
    elif d.gemm_pairs:
        assert L.moe_grouped_gemm_pairs(v.xp, v.cu_seqlens, nseg, v.cap, d.H, 2 * d.I, p(tw[0]), d.E, p(tw[2]),
                                        moe.MOE_EPI_SWIGLU, v.hs, p(st["status"]), None, s) == 0
    else:
        assert L.moe_grouped_gemm(v.xp, v.xp_scales, v.cu_seqlens, nseg, v.cap, d.H, 2 * d.I, p(tw[0]), p(tw[4]),
                                  d.E, p(tw[2]), p(tw[6]), gdt, moe.MOE_EPI_SWIGLU, v.hs, v.hs_scales,
                                  p(st["status"]), s) == 0
    events[3].record()
    if d.fuse_combine:
        # down projection + combine in one launch: the combine stage below is empty
        assert L.moe_grouped_gemm_combine(v.hs, v.hs_scales, v.masked_m if mt else v.cu_seqlens, nseg, mt, v.cap,
                                          d.I, d.H, p(tw[1]), p(tw[5]), d.E, p(tw[3]), p(tw[7]), gdt, v.y, wd_rows,
                                          v.src_row, v.inv_map, None if wd else p(st["wt"]), d.T, d.K, v.shared_map,
                                          p(st["fq"]),
                                          p(st["out"]), v.counters, p(st["status"]), s) == 0
        events[4].record()
        events[5].record()
        return
    if mt:
        assert L.moe_grouped_gemm_batched(v.hs, v.hs_scales, v.masked_m, nseg, mt, d.I, d.H, p(tw[1]), p(tw[5]),
                                          d.E, p(tw[3]), p(tw[7]), gdt, moe.MOE_EPI_NONE, v.y, None,
                                          p(st["status"]), wd_rows, s) == 0
    elif d.gemm_pairs:
        assert L.moe_grouped_gemm_pairs(v.hs, v.cu_seqlens, nseg, v.cap, d.I, d.H, p(tw[1]), d.E, p(tw[3]),
                                        moe.MOE_EPI_NONE, v.y, p(st["status"]), wd_rows, s) == 0
    else:
        assert L.moe_grouped_gemm_ex(v.hs, v.hs_scales, v.cu_seqlens, nseg, v.cap, d.I, d.H, p(tw[1]), p(tw[5]),
                                     d.E, p(tw[3]), p(tw[7]), gdt, moe.MOE_EPI_NONE, v.y, None, p(st["status"]),
                                     wd_rows, s) == 0
    events[4].record()
    if st["fq"] is not None and d.combine_fq_format == 1:
        assert L.moe_combine_nvfp4(v.y, v.inv_map, None if wd else p(st["wt"]), d.T, d.K, d.H,
                                   v.y if d.has_shared else None, v.shared_map, p(st["fq"]), p(st["out"]), s) == 0
    else:
        assert L.moe_combine(v.y, v.inv_map, None if wd else p(st["wt"]), d.T, d.K, d.H,
                             v.y if d.has_shared else None, v.shared_map, p(st["fq"]), p(st["out"]), s) == 0
    events[5].record()


KERNELS_PER_STEP = {"route": 1, "permute": 4, "gemm_gate_up": 1, "gemm_down": 1, "combine": 1}


def algorithmic_work(w, st):
    """Bytes / FLOPs each stage must move or compute for this batch (read once after
    warm-up, outside the timed regions)."""
    lay = st["layer"]
    d = lay.desc
    nseg = d.E + d.has_shared
    if d.max_tokens:
        counts = lay.view("masked_m", (nseg,), torch.int32).cpu().numpy()
    else:
        counts = np.diff(lay.view("cu_seqlens", (nseg + 1,), torch.int32).cpu().numpy())
    n_routed = int(counts[:d.E].sum())
    n_total = int(counts.sum())
    n_tok = int(counts[d.E]) if d.has_shared else int((st["idx"] >= 0).any(dim=1).sum().item())
    T, K, H, I, E = d.T, d.K, d.H, d.I, d.E
    esz = 1 if w.dtype == "e4m3" else 2
    act = H * (1 + 4 / 128) if esz == 1 else H * 2
    experts_touched = int((counts[:E] > 0).sum()) + (1 if d.has_shared else 0)
    return {
        "route": {"bytes": T * E * 4 + T * K * 8},
        "permute": {"bytes": n_tok * H * 2 + n_total * act + T * K * 4 * 2 + lay.views.cap * 4 + T * 4},
        "gemm_gate_up": {"flops": 2.0 * n_total * H * 2 * I, "bytes": experts_touched * 2 * I * H * esz},
        "gemm_down": {"flops": 2.0 * n_total * I * H, "bytes": experts_touched * H * I * esz},
        "combine": {"bytes": (n_routed + (n_total - n_routed)) * H * 2 + T * K * 8 + T * H * 2},
        "_rows": {"n_routed": n_routed, "n_total": n_total, "tokens": n_tok, "experts_touched": experts_touched},
    }


def weight_tiles(args):
    """Whether the layer reads its weights in the tile layout (the SM-pair GEMM reads
    row-major weights only)."""
    return args.weights == "tiles" and not args.gemm_pairs


def run_ours(args, rank, world, local_rank):
    import combine_moe_route_softmax_gb300 as moe
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    w = synth.WORKLOADS[args.workload]
    max_tokens = (args.max_tokens or w.T) if args.layout == "batched" else 0
    st = workload_state(w, rank_seed(0, rank), device, max_tokens, args.fuse_combine, args.dispatch_fq,
                        args.weight_in_down, args.gemm_pairs, weight_tiles(args))
    for _ in range(args.warmup):
        layer_step(st)
    torch.cuda.synchronize()
    assert st["status"].item() == 0, f"device status {st['status'].item()}"
    work = algorithmic_work(w, st)

    # --- timed region 1: the layer with inputs resident in HBM
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            layer_step(st)
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    clocks = clk.summary()

    # --- timed region 2: per-kernel breakdown (same kernels, events between the calls)
    layer_out = st["out"].clone()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        staged_step(st, w, ev[i])
    torch.cuda.synchronize()
    barrier(world)
    # the call-by-call step is the layer's computation: same output bit for bit
    assert torch.equal(st["out"].view(torch.int16), layer_out.view(torch.int16)), "staged step differs from the layer"
    stage_ms = max_stage_times({name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                                for j, name in enumerate(STAGES)}, world, device)

    # --- the layer captured once into a CUDA graph: median of 20 warm replays (no host work
    # per step at all; the workspace and every buffer are fixed, so one capture serves)
    graph_line = None
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg):
        layer_step(st)
    for _ in range(3):
        cg.replay()
    torch.cuda.synchronize()
    reps = []
    for _ in range(20):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        cg.replay()
        b.record()
        reps.append((a, b))
    torch.cuda.synchronize()
    g_ms = max_over_ranks(statistics.median(a.elapsed_time(b) for a, b in reps), world, device)
    assert st["status"].item() == 0, f"device status {st['status'].item()}"
    graph_line = {"median_ms": round(g_ms, 4), "replays": 20,
                  "tokens_per_s": round(w.T_valid * world / (g_ms * 1e-3), 1)}
    del cg

    # --- timed region 3: end to end through moe_layer_forward with host buffers.  A serving
    # pipeline: the next batch's inputs are copied in (pinned host -> device, copy stream)
    # and the previous batch's output copied out (device -> pinned host, a second copy
    # stream) while the current batch computes; input and output buffers are doubled.
    # Only the batch's real tokens cross the host link: the bucket's padding rows (past
    # num_tokens) are never read by the layer and always come out +0, so they stay on the
    # device.
    nv = w.T_valid
    h_logits = st["logits"][:nv].cpu().pin_memory()
    h_x = st["x"][:nv].cpu().pin_memory()
    h_out = [torch.empty((nv, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    d_logits = [torch.zeros_like(st["logits"]) for _ in range(2)]
    d_x = [torch.zeros_like(st["x"]) for _ in range(2)]
    d_out = [torch.empty_like(st["out"]) for _ in range(2)]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def pipeline(n):
        ev = lambda: torch.cuda.Event()
        in_ready, comp_done, out_done = [ev(), ev()], [None, None], [None, None]
        start = torch.cuda.Event(enable_timing=True)
        start.record(comp)
        h2d.wait_event(start)
        d2h.wait_event(start)
        with torch.cuda.stream(h2d):
            d_logits[0][:nv].copy_(h_logits, non_blocking=True)
            d_x[0][:nv].copy_(h_x, non_blocking=True)
            in_ready[0].record(h2d)
        for i in range(n):
            b = i % 2
            comp.wait_event(in_ready[b])
            if out_done[b] is not None:
                comp.wait_event(out_done[b])          # d_out[b] has been copied out
            layer_step(st, x=d_x[b], logits=d_logits[b], out=d_out[b])
            comp_done[b] = ev()
            comp_done[b].record(comp)
            if i + 1 < n:
                nb = (i + 1) % 2
                with torch.cuda.stream(h2d):
                    if comp_done[nb] is not None:
                        h2d.wait_event(comp_done[nb])  # step i-1 no longer reads this input set
                    d_logits[nb][:nv].copy_(h_logits, non_blocking=True)
                    d_x[nb][:nv].copy_(h_x, non_blocking=True)
                    in_ready[nb] = ev()
                    in_ready[nb].record(h2d)
            with torch.cuda.stream(d2h):
                d2h.wait_event(comp_done[b])
                h_out[b].copy_(d_out[b][:nv], non_blocking=True)
                out_done[b] = ev()
                out_done[b].record(d2h)
        for b in range(2):
            if out_done[b] is not None:
                comp.wait_event(out_done[b])
        end = torch.cuda.Event(enable_timing=True)
        end.record(comp)
        return start, end

    pipeline(3)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = pipeline(args.steps)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    assert st["status"].item() == 0
    # the pipelined run's last output reached the host intact (same batch, deterministic kernels)
    assert torch.equal(h_out[(args.steps - 1) % 2], st["out"][:nv].cpu())
    # and the rows that stayed on the device are the bucket's +0 padding
    last = d_out[(args.steps - 1) % 2]
    assert not torch.any(last[nv:].view(torch.int16)), "padding rows of the bucket are not +0"

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    kernels = {}
    for name in STAGES:
        k = {"ms": round(stage_ms[name], 4)}
        if args.fuse_combine and name == "combine":
            # the combine runs inside the down projection's launch: no stage of its own
            k["fused_into"] = "gemm_down"
            kernels[name] = k
            continue
        if args.fuse_combine and name == "gemm_down":
            k["includes"] = "the combine"
        wk = work[name]
        if "flops" in wk:
            k["tflops"] = round(wk["flops"] / (stage_ms[name] * 1e-3) / 1e12, 1)
            k["frac_tc"] = round(k["tflops"] / peaks["bf16_tflops"], 3)
        gbs = wk["bytes"] / (stage_ms[name] * 1e-3) / 1e9
        k["gbs"] = round(gbs, 1)
        k["frac_hbm"] = round(gbs / peaks["hbm_gbs"], 3)
        kernels[name] = k
    dom = max(("gemm_gate_up", "gemm_down"), key=lambda n: stage_ms[n])
    bound = "tensor" if w.dtype == "bf16" else "hbm"
    if bound == "tensor":
        # each GEMM is timed per launch (a few milliseconds between CUDA events), so it is
        # held against the burst tensor peak, not the seconds-long sustained one
        achieved = work[dom]["flops"] / (stage_ms[dom] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
    else:
        achieved = work[dom]["bytes"] / (stage_ms[dom] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        with open(tr_path) as f:
            key = args.workload + ("/batched" if max_tokens else "")
            traffic = json.load(f).get(f"{key}:{dom}")
    cpu = (cpu_baseline(w, tokens=args.cpu_tokens, dispatch_fq=args.dispatch_fq)
           if world == 1 and not args.no_cpu_baseline else None)
    line = {
        "metric": "MoE layer tokens/s at 1 GB300; grouped-GEMM % TC peak; permute/combine % HBM BW",
        "value": round(whole_job_rate(w.T_valid, world, ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "e4m3",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) random-init weights, Zipf(1.1) router bias)",
        "config": {"workload": f"{w.name}: T={w.T_valid} tokens in a {w.T}-row bucket, H={w.H}, I={w.I}, E={w.E}, "
                               f"top-{w.K}, shared={int(w.shared)}, {w.dtype}",
                   "tokens_per_step": w.T_valid, "parallelism": f"token-sharded replicas x{world}",
                   "padding": (f"each slot -1 with p = {w.slot_pad} (the harness masks the routed ids)"
                               if w.slot_pad > 0 else
                               f"bucket rows >= {w.T_valid} (num_tokens on the device)" if w.T_valid < w.T
                               else "none"),
                   "layout": (f"batched [{w.E + int(w.shared)}, {max_tokens}, H] + masked_m" if max_tokens
                              else "contiguous expert-major rows + cu_seqlens"),
                   "combine": ("fused into the down projection" if args.fuse_combine else "separate kernel") +
                              (f", {'NVFP4' if w.fq_format == 'nvfp4' else 'E4M3'} fake-quant at the calibrated "
                               f"constant scale {float(st['fq'].item()):.5g}" if w.fake_quant else ""),
                   "gemm": ("grouped GEMMs on SM pairs (2-SM MMA)" if args.gemm_pairs
                            else "grouped GEMMs one CTA per tile"),
                   "weights": ("tile layout (moe_pack_weights, once at setup, untimed)" if weight_tiles(args)
                               else "row-major [E, N, K]"),
                   "router_weight": ("applied in the down projection's epilogue (weighted rows; the combine sums)"
                                     if args.weight_in_down else "applied in the combine"),
                   "dispatch": (f"{'NVFP4' if args.dispatch_fq == 'nvfp4' else 'E4M3'} fake-quant of the "
                                f"routed experts' rows at the per-tensor scale {float(st['dq'].item()):.5g} "
                                f"({'448 * 6' if args.dispatch_fq == 'nvfp4' else '448'} / max|x|)"
                                if st["dq"] is not None else "rows as they are"),
                   "l2": "no flush: every step streams the weights (far larger than L2) from HBM"},
        "gpu_launches": (sum(KERNELS_PER_STEP.values()) - int(args.fuse_combine)) * args.steps,
        "kernels": kernels,
        "rows": work["_rows"],
        "roofline": {"kernel": dom, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 3), "traffic": traffic,
                     "peak_source": f"{peak_src} ({'bf16_tflops' if bound == 'tensor' else 'hbm_gbs'})"},
        "e2e": {"value": round(whole_job_rate(w.T_valid, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h_logits.numel() * 4 + h_x.numel() * 2,
                "d2h_bytes_per_step": h_out[0].numel() * 2,
                "pipeline": "inputs of step i+1 copied in and output of step i-1 copied out during step i; "
                            "only the batch's real tokens cross the host link (bucket padding stays on the "
                            "device)"},
        "graph": graph_line,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    emit(line, rank)


# ------------------------------------------------------------------- CPU oracle arm
def oracle_sample(w, tokens, seed=0):
    """Inputs for the oracle on a sample of the workload's tokens (host, untimed): the
    sample's logits and activations and the BF16 weights of every expert it routes to."""
    from oracle import moe_ref as ref
    logits = synth.router_logits(w, seed).numpy()
    x = synth.hidden(w, seed)
    toks = np.arange(tokens)
    idx, _ = ref.route_topk(logits[toks], w.K)
    experts = sorted(set(idx.reshape(-1).tolist()))
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    w13 = {e: bits(synth.expert_w13(w, 0, e)) for e in experts}
    w2 = {e: bits(synth.expert_w2(w, 0, e)) for e in experts}
    shared = (bits(synth.expert_w13(w, 0, w.E)), bits(synth.expert_w2(w, 0, w.E))) if w.shared else None
    return logits[toks], bits(x[:tokens]), w13, w2, shared


def oracle_step(w, sample, per_call=None, dispatch_fq=None):
    """The oracle's layer on the sample: route, permute, fp64 experts and the sum (per-call
    seconds accumulated into `per_call` when given).  dispatch_fq (None, "e4m3" or "nvfp4"):
    the routed experts see the sample's rows fake-quantised in that format at the oracle's
    own per-tensor scale."""
    from oracle import moe_ref as ref
    logits, xb, w13, w2, shared = sample
    t0 = time.perf_counter()
    idx, wt = ref.route_topk(logits, w.K)
    t1 = time.perf_counter()
    ref.permute(idx, w.E, with_shared=w.shared)
    t2 = time.perf_counter()
    dq = None
    if dispatch_fq:
        a = ref.tensor_amax(xb)
        dq = ref.nvfp4_scale_from_amax(a) if dispatch_fq == "nvfp4" else ref.fq_scale_from_amax(a)
    out = ref.layer_reference(xb, idx, wt, w13, w2, shared=shared, dispatch_scale=dq,
                              dispatch_format=dispatch_fq or "e4m3")
    t3 = time.perf_counter()
    if per_call is not None:
        for k, v in (("route", t1 - t0), ("permute", t2 - t1), ("experts_and_sum", t3 - t2)):
            per_call[k] = per_call.get(k, 0.0) + v
    return out


def cpu_baseline(w, tokens=8, reps=1, dispatch_fq=None):
    sample = oracle_sample(w, tokens)
    per_call = {}
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(w, sample, per_call, dispatch_fq)
    dt = (time.perf_counter() - t0) / reps
    return {"value": round(tokens / dt, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{tokens} tokens of the {w.name} workload through the numpy oracle (route, permute, fp64 "
                      f"experts, fixed-order sum); {dt:.1f} s",
            "per_call_s": {k: round(v / reps, 4) for k, v in per_call.items()}}


def run_reference(args, rank, world):
    dist_init(world, "gloo")
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    sample = oracle_sample(w, args.ref_tokens)
    for _ in range(args.warmup):
        oracle_step(w, sample, None, args.dispatch_fq)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, sample, None, args.dispatch_fq)
    dt = (time.perf_counter() - t0) / args.steps
    v = round(args.ref_tokens / dt, 3)
    line = {
        "impl": "reference",
        "metric": "MoE layer tokens/s at 1 GB300; grouped-GEMM % TC peak; permute/combine % HBM BW",
        "value": v, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"{w.name}: T={w.T_valid} tokens in a {w.T}-row bucket, H={w.H}, I={w.I}, E={w.E}, "
                               f"top-{w.K}, shared={int(w.shared)}, {w.dtype}",
                   "tokens_per_step": args.ref_tokens,
                   "dispatch": (f"{'NVFP4' if args.dispatch_fq == 'nvfp4' else 'E4M3'} fake-quant of the routed "
                                f"experts' rows at a per-tensor scale from max|x|" if args.dispatch_fq
                                else "rows as they are")},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "kind": "oracle", "cores": os.cpu_count(),
                         "sample": f"{args.ref_tokens} tokens per step through the numpy oracle"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, rank)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=64)
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layout", choices=["contiguous", "batched"], default="contiguous",
                    help="expert-major rows with cu_seqlens, or the batched [E, max_tokens, H] layout")
    ap.add_argument("--weight-in-down", action="store_true",
                    help="apply the router weights in the down projection's epilogue (the combine only sums)")
    ap.add_argument("--dispatch-fq", nargs="?", const="e4m3", default=None, choices=["e4m3", "nvfp4"],
                    help="BF16 workloads: fake-quant of the routed experts' input rows, E4M3 (default) or NVFP4, "
                         "at a per-tensor scale from the batch's amax")
    ap.add_argument("--gemm-pairs", action="store_true",
                    help="BF16: both grouped GEMMs on SM pairs with the 2-SM MMA (moe_grouped_gemm_pairs)")
    ap.add_argument("--fuse-combine", action="store_true",
                    help="run the combine inside the down projection (moe_grouped_gemm_combine)")
    ap.add_argument("--weights", choices=["tiles", "rows"], default="tiles",
                    help="expert weights in the tile layout of moe_pack_weights (default; not with --gemm-pairs, "
                         "which reads row-major weights) or row-major")
    ap.add_argument("--max-tokens", type=int, default=0,
                    help="rows per expert block of the batched layout (default: the bucket's T, which never "
                         "overflows)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rc = launch_ranks(args.gpus, sys.argv[1:])
    if rc is not None:
        sys.exit(rc)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
