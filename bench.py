#!/usr/bin/env python
"""Benchmark of the prefix-cached KV attention hot path on GB300.

Headline line (one JSON object on stdout): the GQA decode workload over an mlx4g32 prefix --
16 layers, H_q=32, H_kv=8, D=64, N=8192, M=1, fused dense suffix S_suf=16. One step is one
decode step of the model's attention: all 16 layers' prefix + suffix attention, issued as one
batched launch of the split-K decode kernel. Inputs are resident in HBM when the timed region
starts; the step rotates over 4 distinct prefix sets (4 x 84 MB, more than the L2 size the
device reports) so that no step reads data left in L2 by the previous three. ``value`` is
prefix KV record bytes per second.

Extra keys report the other rows of the hot path (the same workload as 16 dependent per-layer
calls, fp16 M=1 at D=128 and at the other head dimensions, batched-Q prefill over fp16 and
mlx4g32 prefixes, sparse top-K, cartridge quantise + dequantise + 64-session attend), each with
its own roofline fraction.

``--impl reference`` times the CPU oracle (test infrastructure) on all the host cores on the
same workload and prints the same line with ``"impl": "reference"``. ``--profile ROW`` runs each
kernel of one row once, at a size meant for an Nsight Compute capture, and prints nothing else.
"""
import os

# Each CPU oracle process (reference arm / cpu_baseline) runs single-threaded, one per host core,
# so the core count is known.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefix-attn KV bytes/s at M=1, TFLOP/s at M=512; % of GB300 roofline"
WORKLOAD = "gqa_decode_mlx4g32"
W = dict(H_q=32, H_kv=8, N=8192, D=64, layers=16, S_suf=16)
REC_BYTES = W["H_kv"] * W["D"] // 2 + W["H_kv"] * W["D"] // 8        # 320 B / token / side
KV_BYTES_STEP = W["layers"] * 2 * W["N"] * REC_BYTES                     # 83,886,080
SUF_BYTES_STEP = W["layers"] * 2 * W["H_kv"] * W["S_suf"] * W["D"] * 2
Q_BYTES_STEP = W["layers"] * W["H_q"] * W["D"] * 4
O_BYTES_STEP = W["layers"] * (W["H_q"] * W["D"] * 4 + W["H_q"] * 4)
ALG_BYTES_STEP = KV_BYTES_STEP + SUF_BYTES_STEP + Q_BYTES_STEP + O_BYTES_STEP
ROTATE = 4


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p.get("bf16_tflops_sustained"), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def traffic_from_profiles(name):
    """dram bytes per launch recorded from an ncu capture (profiles/<name>.txt), or None."""
    path = os.path.join(ROOT, "profiles", name + ".txt")
    try:
        for line in open(path):
            if line.startswith("traffic_bytes_per_launch:"):
                v = line.split(":", 1)[1].strip()
                return None if v in ("", "null") else float(v)
    except OSError:
        pass
    return None


# ------------------------------------------------------------------ clocks during the timed region

class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            time.sleep(0.2)
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        rows = []
        for ln in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) >= 7:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ helpers (GPU arm)

def _torch():
    import torch
    return torch


def flush_l2(buf):
    buf.add_(1)


class Timer:
    """CUDA events on the stream the library launches on (torch's current stream)."""

    def __init__(self, n):
        torch = _torch()
        self.s = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        self.e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    def ms(self):
        _torch().cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(self.s, self.e)]


def setup_decode_sets(ctx, torch, seed=0):
    """ROTATE distinct sets of 16 mlx4g32 layers + per-layer Q, suffix, outputs (device). A set's
    per-layer inputs (Q, K_suf, V_suf) are views into one device buffer and its outputs (O, then
    LSE) into another, the way a serving loop keeps one step's inputs together: the end-to-end
    path then moves each step's inputs and results with one copy each way."""
    H_q, H_kv, N, D, L, S = W["H_q"], W["H_kv"], W["N"], W["D"], W["layers"], W["S_suf"]
    from prefix_cached_kv_gb300 import synth
    q_b, s_b, o_b, l_b = H_q * D * 4, H_kv * S * D * 2, H_q * D * 4, H_q * 4
    per_in = q_b + 2 * s_b
    sets, arenas = [], []
    for r in range(ROTATE):
        din = torch.empty(L * per_in, dtype=torch.uint8, device="cuda")
        dout = torch.empty(L * (o_b + l_b), dtype=torch.uint8, device="cuda")
        descs = []
        for layer in range(L):
            K, V = synth.torch_gen_kv_device(seed + 101 * r, H_kv, N, D, "cuda", col_scale=True, layer=layer)
            ctx.store(f"bench{r}", layer, K, V, fmt=1)
            g = torch.Generator(device="cuda").manual_seed(1000 * r + layer)
            base = layer * per_in
            Q = din[base:base + q_b].view(torch.float32).view(H_q, D)
            Ks = din[base + q_b:base + q_b + s_b].view(torch.float16).view(H_kv, S, D)
            Vs = din[base + q_b + s_b:base + per_in].view(torch.float16).view(H_kv, S, D)
            Q.copy_(torch.randn((H_q, D), generator=g, device="cuda"))
            Ks.copy_(torch.randn((H_kv, S, D), generator=g, device="cuda").half())
            Vs.copy_(torch.randn((H_kv, S, D), generator=g, device="cuda").half())
            O = dout[layer * o_b:(layer + 1) * o_b].view(torch.float32).view(H_q, D)
            LSE = dout[L * o_b + layer * l_b:L * o_b + (layer + 1) * l_b].view(torch.float32)
            descs.append(dict(sid=f"bench{r}", layer=layer, Q=Q, O=O, LSE=LSE, K_suf=Ks, V_suf=Vs))
        sets.append(descs)
        arenas.append((din, dout))
    torch.cuda.synchronize()
    return sets, arenas


def graph_of(torch, fn):
    """Capture fn() (library calls on the current stream) into a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=st):
        fn()
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    return g


def time_replays(torch, g, n):
    """Events around n back-to-back replays of g on the current stream -> ms per replay."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def run_main(args, ctx, torch, pk):
    sets, arenas = setup_decode_sets(ctx, torch)
    H_q, H_kv, D, S = W["H_q"], W["H_kv"], W["D"], W["S_suf"]
    callers = [ctx.batch_caller(sets[r], H_q, H_kv, D, S_suf=S) for r in range(ROTATE)]
    for c in callers:          # eager warm-up (first launch sets kernel attributes)
        c()
    torch.cuda.synchronize()
    # one graph replay = ROTATE steps, one per distinct prefix set (each step one kernel launch)
    g = graph_of(torch, lambda: [c() for c in callers])
    reps = max(1, (args.steps + ROTATE - 1) // ROTATE)
    steps = reps * ROTATE
    with ClockSampler(torch.cuda.current_device()) as cs:
        t_end = time.perf_counter() + 0.6          # warm-up: >= W steps and >= 0.6 s under load
        n = 0
        while n < args.warmup or time.perf_counter() < t_end:
            g.replay()
            n += ROTATE
            if n % 400 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        ms_rep = time_replays(torch, g, reps)
        barrier()
    ms_step = max_over_ranks(ms_rep / ROTATE)
    ctx.sync()
    clocks = cs.summary()
    clocks["window"] = "timed region + >= 0.6 s of identical warm-up steps just before it"
    achieved = ALG_BYTES_STEP / (ms_step * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm"], 4), "traffic": traffic_from_profiles("decode_mlx4g32_gqa"),
            "kernel": "decode_kernel<mlx4g32, D=64> + merge_kernel", "algorithmic_bytes_per_launch": ALG_BYTES_STEP,
            "duration": "per-step time of back-to-back graph-replayed steps (decode + merge, PDL-chained)",
            "peak_source": f"{pk['src']} hbm_gbs"}
    latency = run_latency(args, ctx, torch, sets, pk)
    e2e = run_e2e(args, ctx, torch, sets, arenas)
    return ms_step, steps, clocks, roof, e2e, latency


def run_latency(args, ctx, torch, sets, pk):
    """The same step as a model's decode runs it: 16 dependent per-layer pck_query_fused calls
    (each a decode + merge), one CUDA graph per prefix set, rotating over the 4 sets."""
    H_q, H_kv, D = W["H_q"], W["H_kv"], W["D"]

    def step(r):
        for d in sets[r]:
            ctx.query_fused(d["sid"], d["layer"], d["Q"].view(H_q, 1, D), d["K_suf"], d["V_suf"],
                            O=d["O"].view(H_q, 1, D), LSE=d["LSE"].view(H_q, 1))

    for r in range(ROTATE):
        step(r)
    torch.cuda.synchronize()
    g = graph_of(torch, lambda: [step(r) for r in range(ROTATE)])
    for _ in range(max(3, args.warmup)):
        g.replay()
    reps = 50
    ms = time_replays(torch, g, reps) / ROTATE
    ctx.sync()
    gbs = ALG_BYTES_STEP / (ms * 1e-3) / 1e9
    return {"workload": WORKLOAD + " as 16 dependent per-layer fused calls (latency mode)",
            "us_per_step": round(ms * 1e3, 2), "us_per_layer": round(ms * 1e3 / W["layers"], 3),
            "record_gbs": round(KV_BYTES_STEP / (ms * 1e-3) / 1e9, 1), "frac_hbm": round(gbs / pk["hbm"], 4),
            "launches_per_step": 2 * W["layers"], "steps_timed": reps * ROTATE}


def run_e2e(args, ctx, torch, sets, arenas):
    """The headline step end to end through the host-buffer call: each step's Q and suffixes sit in
    pinned host memory and O, LSE land there; pck_query_batch_host moves the bytes (a copy kernel
    pulls the inputs over the host link into device staging, the merge writes O and LSE into the
    host buffers)."""
    H_q, H_kv, D, S = W["H_q"], W["H_kv"], W["D"], W["S_suf"]
    # pinned host arenas with the device arenas' layout (one step's inputs, one step's outputs)
    hosts = [(din.cpu().pin_memory(), torch.empty(dout.shape, dtype=dout.dtype).pin_memory()) for din, dout in arenas]
    h2d = arenas[0][0].numel()
    d2h = arenas[0][1].numel()

    def host_view(t, dev_arena, host_arena):
        off = t.data_ptr() - dev_arena.data_ptr()
        return host_arena[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    calls = []
    for r in range(ROTATE):
        (din, dout), (hin, hout) = arenas[r], hosts[r]
        hd = [dict(sid=d["sid"], layer=d["layer"], Q=host_view(d["Q"], din, hin), O=host_view(d["O"], dout, hout),
                   LSE=host_view(d["LSE"], dout, hout), K_suf=host_view(d["K_suf"], din, hin),
                   V_suf=host_view(d["V_suf"], din, hin)) for d in sets[r]]
        calls.append(ctx.batch_caller(hd, H_q, H_kv, D, S_suf=S, host=True))
    for c in calls:   # eager once (first calls set kernel attributes), then capture
        c()
    torch.cuda.synchronize()
    # a serving loop's step: the call as one CUDA graph per input set, one launch and one stream
    # synchronize per step
    graphs = [graph_of(torch, c) for c in calls]

    def step(k):
        graphs[k % ROTATE].replay()
        torch.cuda.current_stream().synchronize()

    n_steps = min(args.steps, 400)
    for k in range(max(args.warmup, 3)):
        step(k)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(n_steps):
        step(k)
    dt = max_over_ranks((time.perf_counter() - t0) * 1e3)
    return {"value": round(job_throughput(KV_BYTES_STEP * n_steps, dt) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(dt / n_steps, 4),
            "steps": n_steps, "path": "pinned host Q + suffixes of the 16 layers -> pck_query_batch_host (a copy "
                                      "kernel reads them over the host link into device staging; the merge kernel "
                                      "writes O + LSE into the pinned host buffers), captured as one CUDA graph per "
                                      "input set; one graph launch and one stream synchronize every step"}


# ------------------------------------------------------------------ other rows of the hot path

def row_fp16_m1(ctx, torch, pk, reps=20):
    """Single-layer fp16 M=1 (H=8, N=2048, D=128) over 64 distinct sessions (537 MB > L2):
    64 single-session calls back to back (per-call time), and the 64 as one batched launch."""
    from prefix_cached_kv_gb300 import synth
    H, N, D, R = 8, 2048, 128, 64
    for r in range(R):
        K, V = synth.torch_gen_kv_device(7 + r, H, N, D, "cuda", col_scale=True)
        ctx.store(f"f16m1_{r}", 0, K, V)
    Qs = [torch.randn((H, 1, D), device="cuda") for _ in range(R)]
    Os = [torch.empty((H, 1, D), device="cuda") for _ in range(R)]
    Ls = [torch.empty((H, 1), device="cuda") for _ in range(R)]
    kv = 2 * H * N * D * 2
    singles = lambda: [ctx.query(f"f16m1_{r}", 0, Qs[r], O=Os[r], LSE=Ls[r]) for r in range(R)]
    singles()
    g1 = graph_of(torch, singles)
    for _ in range(3):
        g1.replay()
    lat = time_replays(torch, g1, reps) / R
    descs = [dict(sid=f"f16m1_{r}", layer=0, Q=Qs[r][:, 0], O=Os[r][:, 0], LSE=Ls[r][:, 0]) for r in range(R)]
    call = ctx.batch_caller(descs, H, H, D)
    call()
    g2 = graph_of(torch, call)
    for _ in range(3):
        g2.replay()
    thr = time_replays(torch, g2, reps)
    ctx.sync()
    for r in range(R):
        ctx.drop(f"f16m1_{r}")
    gbs = R * kv / (thr * 1e-3) / 1e9
    return {"workload": "prefix_m1_fp16 H=8 N=2048 D=128", "us_per_call_back_to_back": round(lat * 1e3, 2),
            "kv_gbs_single_calls": round(kv / (lat * 1e-3) / 1e9, 1),
            "frac_hbm_single_calls": round(kv / (lat * 1e-3) / 1e9 / pk["hbm"], 4),
            "kv_gbs_64_sessions_one_launch": round(gbs, 1), "frac_hbm_64_sessions": round(gbs / pk["hbm"], 4)}


def row_dims(ctx, torch, pk, reps=20):
    """fp16 M=1 at the other head dimensions (D = 32, 96, 160, 192, 256, 512): 64 sessions of H=8
    in one batched launch, N = 262,144 / D tokens so every session holds 8.4 MB of K/V whatever D
    (537 MB per pass, over 4x L2)."""
    from prefix_cached_kv_gb300 import synth
    H, R = 8, 64
    out = {"workload": "prefix_m1_fp16 at other head dims, 64 sessions x H=8 in one launch"}
    for D in (32, 96, 160, 192, 256, 512):
        N = 262144 // D
        for r in range(R):
            K, V = synth.torch_gen_kv_device(11 + r, H, N, D, "cuda", col_scale=True)
            ctx.store(f"dims_{r}", 0, K, V)
        Qs = [torch.randn((H, D), device="cuda") for _ in range(R)]
        Os = [torch.empty((H, D), device="cuda") for _ in range(R)]
        Ls = [torch.empty((H,), device="cuda") for _ in range(R)]
        descs = [dict(sid=f"dims_{r}", layer=0, Q=Qs[r], O=Os[r], LSE=Ls[r]) for r in range(R)]
        call = ctx.batch_caller(descs, H, H, D)
        call()
        g = graph_of(torch, call)
        for _ in range(3):
            g.replay()
        ms = time_replays(torch, g, reps)
        ctx.sync()
        del g
        for r in range(R):
            ctx.drop(f"dims_{r}")
        gbs = R * 2 * H * N * D * 2 / (ms * 1e-3) / 1e9
        out[f"D{D}_kv_gbs"] = round(gbs, 1)
        out[f"D{D}_frac_hbm"] = round(gbs / pk["hbm"], 4)
    return out


def row_sparse(ctx, torch, pk, reps=10, l2=None):
    """Sparse top-K (N=65,536, D=256, H_q=8, H_kv=2, B=64, K_top=8, S_suf=32) with the seeded
    needles. Single-query mode: one query call per session back to back over 64 sessions (four
    kernels a call). Throughput mode: 64 sessions (the batch limit) per pck_query_sparse_batch
    call (one fused kernel, 128 CTAs), rotating over enough distinct 64-session sets that the
    bytes one pass touches exceed 4x the L2 size. Bytes counted: block means + selected K/V + suffix + Q/O (not the dense
    prefix)."""
    from prefix_cached_kv_gb300 import synth
    H_q, H_kv, N, D, B, Kt, S, R = 8, 2, 65536, 256, 64, 8, 32, 64
    nbk = N // B
    alg = H_kv * nbk * D * 4 + 8 * B * D * 2 * 2 * H_kv + 2 * H_kv * S * D * 2 + H_q * D * 4 * 2 + H_q * 4
    l2 = l2 or (126 << 20)
    n_sets = max(1, -(-4 * l2 // (R * alg)))         # ceil(4 L2 / bytes of one set)
    hm = synth.default_head_map(H_q, H_kv)
    K, V = synth.gen_kv(0, H_kv, N, D)
    Q = synth.gen_q(0, H_q, 1, D)[:, 0]
    needles = synth.needle_blocks(0, N // B, Kt)
    K = synth.plant_needles(K, Q, hm, needles, B)
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    Kd, Vd = dv(K), dv(V)
    n_sess = n_sets * R
    for r in range(n_sess):
        ctx.store(f"sparse{r}", 0, Kd, Vd)
        ctx.build_block_means(f"sparse{r}", 0, B)
    del Kd, Vd
    # every session reads its own copy of Q (the needles were planted toward this Q) and its own suffix
    Qd = dv(Q)
    Qs = [Qd.clone() for _ in range(n_sess)]
    Kss = [torch.randn((H_kv, S, D), device="cuda").half() for _ in range(n_sess)]
    Vss = [torch.randn((H_kv, S, D), device="cuda").half() for _ in range(n_sess)]
    Os = [torch.empty((H_q, D), device="cuda") for _ in range(n_sess)]
    Ls = [torch.empty((H_q,), device="cuda") for _ in range(n_sess)]
    idx = [torch.empty((H_q, Kt), dtype=torch.int32, device="cuda") for _ in range(n_sess)]
    calls = lambda: [ctx.query_sparse_auto(f"sparse{r}", 0, Qs[r], B, Kt, H_kv, K_suf=Kss[r], V_suf=Vss[r], O=Os[r],
                                           LSE=Ls[r], idx=idx[r]) for r in range(R)]
    calls()
    g = graph_of(torch, calls)
    for _ in range(3):
        g.replay()
    ms = time_replays(torch, g, reps) / R
    ctx.sync()
    ok = all(bool((t.cpu().numpy() == needles[None]).all()) for t in idx[:R])
    del g
    for t in idx:
        t.fill_(-1)
    bcalls = []
    for k in range(n_sets):
        descs = [dict(sid=f"sparse{r}", layer=0, Q=Qs[r], O=Os[r], LSE=Ls[r], K_suf=Kss[r], V_suf=Vss[r], idx=idx[r])
                 for r in range(k * R, (k + 1) * R)]
        bcalls.append(ctx.sparse_batch_caller(descs, H_q, H_kv, D, B, Kt, S_suf=S))
    for c in bcalls:
        c()
    gb = graph_of(torch, lambda: [c() for c in bcalls])
    for _ in range(3):
        gb.replay()
    ms_b = time_replays(torch, gb, reps) / n_sess
    ctx.sync()
    ok_b = all(bool((t.cpu().numpy() == needles[None]).all()) for t in idx)
    del gb
    for r in range(n_sess):
        ctx.drop(f"sparse{r}")
    gbs = lambda t_ms: alg / (t_ms * 1e-3) / 1e9
    return {"workload": "sparse_topk_64k", "us_per_call_back_to_back": round(ms * 1e3, 2),
            "alg_bytes_per_call": alg, "gbs": round(gbs(ms), 1), "frac_hbm": round(gbs(ms) / pk["hbm"], 4),
            "needles_selected": ok, "launches_per_call": 4, "batched_launches_per_call": 1,
            "batched_form": "one fused kernel, a CTA per (session, kv head): scores on the tensor cores, top-K, union, gather decode, merge",
            "batched_sessions_per_call": R, "batched_sets_rotated": n_sets,
            "batched_touched_mb_per_pass": round(n_sess * alg / 1e6, 1), "l2_mb": round(l2 / 1e6, 1),
            "batched_us_per_session": round(ms_b * 1e3, 3),
            "batched_gbs": round(gbs(ms_b), 1), "batched_frac_hbm": round(gbs(ms_b) / pk["hbm"], 4),
            "batched_needles_selected": ok_b}


def row_cartridge(ctx, torch, pk, reps=10):
    """Cartridge: quantise 86,580 tokens x 36 layers x (K, V) at kv_dim 1024 in one launch (read
    12.77 GB fp16, write 3.99 GB records); then 64 sessions' M=1 GQA queries over their 8192-token
    windows (mlx4g32) in one launch (671 MB of records, > L2)."""
    from prefix_cached_kv_gb300 import binding, synth
    N, L, kv, Wn, S = 86580, 36, 1024, 8192, 64
    H_q, H_kv, D = 32, 8, 128
    rows = N * L * 2
    X = torch.empty((rows, kv), dtype=torch.float16, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    for i in range(0, rows, N):
        X[i:i + N].normal_(generator=g)
    rec = torch.empty((rows, kv // 2 + kv // 8), dtype=torch.uint8, device="cuda")
    binding.quantize_mlx4g32(X, rec)
    torch.cuda.synchronize()
    tm = Timer(reps)
    for k in range(reps):
        tm.s[k].record()
        binding.quantize_mlx4g32(X, rec)
        tm.e[k].record()
    qms = statistics.median(tm.ms())
    qbytes = rows * kv * 2 + rows * (kv // 2 + kv // 8)
    del X
    # WARM / FETCH RANGE form of every stored record: [8, rows, 128] fp16 (dequantise + transpose)
    Y = torch.empty((8, rows, kv // 8), dtype=torch.float16, device="cuda")
    binding.dequantize_mlx4g32(rec, rows, 8, kv // 8, out=Y)
    torch.cuda.synchronize()
    tm = Timer(reps)
    for k in range(reps):
        tm.s[k].record()
        binding.dequantize_mlx4g32(rec, rows, 8, kv // 8, out=Y)
        tm.e[k].record()
    wms = statistics.median(tm.ms())
    wbytes = rows * (kv // 2 + kv // 8) + rows * kv * 2
    del Y
    rb = kv // 2 + kv // 8
    descs = []
    for s in range(S):
        layer = s % L
        o = synth.cartridge_window_start(s, N, Wn)
        kbase = (layer * 2) * N + o
        vbase = (layer * 2 + 1) * N + o
        ctx.store_records(f"cart{s}", 0, H_kv, Wn, D, rec[kbase:kbase + Wn], rec[vbase:vbase + Wn])
        descs.append(dict(sid=f"cart{s}", layer=0, Q=torch.randn((H_q, D), device="cuda"),
                          O=torch.empty((H_q, D), device="cuda"), LSE=torch.empty((H_q,), device="cuda")))
    del rec
    call = ctx.batch_caller(descs, H_q, H_kv, D)
    call()
    ga = graph_of(torch, call)
    for _ in range(3):
        ga.replay()
    ams = time_replays(torch, ga, reps)
    ctx.sync()
    for s in range(S):
        ctx.drop(f"cart{s}")
    abytes = S * Wn * 2 * rb
    return {"workload": "cartridge_mlx4g32",
            "quantize_ms": round(qms, 3), "quantize_gbs": round(qbytes / (qms * 1e-3) / 1e9, 1),
            "quantize_frac_hbm": round(qbytes / (qms * 1e-3) / 1e9 / pk["hbm"], 4),
            "quantize_tokens_per_s": round(N * L / (qms * 1e-3), 0),
            "warm_dequantize_ms": round(wms, 3), "warm_dequantize_gbs": round(wbytes / (wms * 1e-3) / 1e9, 1),
            "warm_dequantize_frac_hbm": round(wbytes / (wms * 1e-3) / 1e9 / pk["hbm"], 4),
            "warm_bytes": wbytes,
            "attend_us": round(ams * 1e3, 2), "attend_kv_gbs": round(abytes / (ams * 1e-3) / 1e9, 1),
            "attend_frac_hbm": round(abytes / (ams * 1e-3) / 1e9 / pk["hbm"], 4)}


def row_prefill(ctx, torch, pk, reps=10, fmt=0):
    """Batched-Q prefill: 28 layers, H_q=24, H_kv=8, D=128, N=4096 prefix (fp16, or mlx4g32 with
    fmt=1), M=512 fp16 queries, causal S_suf=512 suffix; algorithmic FLOPs count only unmasked
    scores at head dimension D (the mlx4g32 form's hi/lo pairs double the tensor-core work)."""
    from prefix_cached_kv_gb300 import binding
    H_q, H_kv, D, N, M, S, L = 24, 8, 128, 4096, 512, 512, 28
    flops_layer = 4 * H_q * M * N * D + 4 * H_q * D * (M * (M + 1) // 2)
    name = "batched_q_prefill" + ("" if fmt == 0 else " over an mlx4g32 prefix")
    try:
        for layer in range(L):
            K = torch.randn((H_kv, N, D), device="cuda").half()
            V = torch.randn((H_kv, N, D), device="cuda").half()
            ctx.store("prefill", layer, K, V, fmt=fmt)
        Qs = [torch.randn((H_q, M, D), device="cuda").half() for _ in range(L)]
        Ks = [torch.randn((H_kv, S, D), device="cuda").half() for _ in range(L)]
        Vs = [torch.randn((H_kv, S, D), device="cuda").half() for _ in range(L)]
        O = torch.empty((H_q, M, D), device="cuda")
        LSE = torch.empty((H_q, M), device="cuda")
        ctx.query_fused("prefill", 0, Qs[0], Ks[0], Vs[0], O=O, LSE=LSE)
    except binding.PckError as e:
        for layer in range(L):
            ctx.drop("prefill", layer)
        return {"workload": name, "unavailable": str(e)}
    # one graph replay = the L layer calls back to back (staging + kernel + merge each), so the
    # GPU time is measured without the host's per-call launch cost in between
    g = graph_of(torch, lambda: [ctx.query_fused("prefill", l, Qs[l], Ks[l], Vs[l], O=O, LSE=LSE) for l in range(L)])
    for _ in range(3):
        g.replay()
    n_rep = max(3, reps // L)
    ms = statistics.median(time_replays(torch, g, 1) for _ in range(n_rep)) / L
    ctx.sync()
    del g
    for layer in range(L):
        ctx.drop("prefill", layer)
    tf = flops_layer / (ms * 1e-3) / 1e12
    return {"workload": name, "ms_per_layer": round(ms, 4), "tflops": round(tf, 1),
            "frac_tensor_bf16_peak": round(tf / pk["bf16"], 4), "gflop_per_layer": round(flops_layer / 1e9, 3)}


# ------------------------------------------------------------------ single launches for Nsight Compute

def profile_row(row, ctx, torch):
    """Run each kernel of one row twice (the first launch sets kernel attributes; capture the
    second with -s / -c), at sizes that keep a capture to a few GB on the device: fp16 = the
    64-session fp16 M=1 batch; sparse = a 16-session pck_query_sparse_batch (scoring, selection,
    gather decode, merge); quant = one cartridge layer's K and V (354 MB in); warm = the same
    layer's records dequantised to fp16; prefill = one batched-Q layer (fp16 prefix);
    prefill_mlx = the same over an mlx4g32 prefix."""
    from prefix_cached_kv_gb300 import binding, synth
    if row == "fp16":
        H, N, D, R = 8, 2048, 128, 64
        descs = []
        for r in range(R):
            K, V = synth.torch_gen_kv_device(7 + r, H, N, D, "cuda", col_scale=True)
            ctx.store(f"pf{r}", 0, K, V)
            descs.append(dict(sid=f"pf{r}", layer=0, Q=torch.randn((H, D), device="cuda"),
                              O=torch.empty((H, D), device="cuda"), LSE=torch.empty((H,), device="cuda")))
        fn = lambda: ctx.query_batch(descs, H, H, D)
    elif row == "sparse":
        H_q, H_kv, N, D, B, Kt, S, R = 8, 2, 65536, 256, 64, 8, 32, 16
        hm = synth.default_head_map(H_q, H_kv)
        K, V = synth.gen_kv(0, H_kv, N, D)
        Q = synth.gen_q(0, H_q, 1, D)[:, 0]
        K = synth.plant_needles(K, Q, hm, synth.needle_blocks(0, N // B, Kt), B)
        dv = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        Kd, Vd, Qd = dv(K), dv(V), dv(Q)
        Ks, Vs = [dv(a) for a in synth.gen_suffix(0, H_kv, S, D)]
        descs = []
        for r in range(R):
            ctx.store(f"ps{r}", 0, Kd, Vd)
            ctx.build_block_means(f"ps{r}", 0, B)
            descs.append(dict(sid=f"ps{r}", layer=0, Q=Qd, O=torch.empty((H_q, D), device="cuda"),
                              LSE=torch.empty((H_q,), device="cuda"), K_suf=Ks, V_suf=Vs,
                              idx=torch.empty((H_q, Kt), dtype=torch.int32, device="cuda")))
        fn = ctx.sparse_batch_caller(descs, H_q, H_kv, D, B, Kt, S_suf=S)
    elif row in ("quant", "warm"):
        N, kv = 86580, 1024
        X = synth.torch_gen_rows_device(0, 2 * N, kv, "cuda", stream=1)
        rec = binding.quantize_mlx4g32(X)
        if row == "quant":
            fn = lambda: binding.quantize_mlx4g32(X, rec)
        else:
            Y = torch.empty((8, 2 * N, 128), dtype=torch.float16, device="cuda")
            fn = lambda: binding.dequantize_mlx4g32(rec, 2 * N, 8, 128, out=Y)
    elif row in ("prefill", "prefill_mlx"):
        H_q, H_kv, D, N, M, S = 24, 8, 128, 4096, 512, 512
        ctx.store("pp", 0, torch.randn((H_kv, N, D), device="cuda").half(),
                  torch.randn((H_kv, N, D), device="cuda").half(), fmt=0 if row == "prefill" else 1)
        Q = torch.randn((H_q, M, D), device="cuda").half()
        Ks = torch.randn((H_kv, S, D), device="cuda").half()
        Vs = torch.randn((H_kv, S, D), device="cuda").half()
        fn = lambda: ctx.query_fused("pp", 0, Q, Ks, Vs)
    else:
        raise SystemExit(f"unknown profile row {row}")
    torch.cuda.synchronize()
    for _ in range(2):
        fn()
        torch.cuda.synchronize()
    ctx.sync()


# ------------------------------------------------------------------ CPU oracle (reference arm, cpu_baseline)

def oracle_layer_inputs(layer, seed=0):
    """Host inputs of one layer of the headline workload, records built by the oracle's quantiser
    (store side, not timed)."""
    from oracle import pck_oracle as orc
    from prefix_cached_kv_gb300 import synth
    H_q, H_kv, N, D, S = W["H_q"], W["H_kv"], W["N"], W["D"], W["S_suf"]
    K, V = synth.gen_kv(seed, H_kv, N, D, layer=layer)
    tok = lambda X: X.transpose(1, 0, 2).reshape(N, H_kv * D)
    return dict(Krec=orc.quantize_records(tok(K)), Vrec=orc.quantize_records(tok(V)),
                Q=synth.gen_q(seed, H_q, 1, D, layer=layer), suf=synth.gen_suffix(seed, H_kv, S, D, layer=layer))


def oracle_layer(inp, n_tok=None):
    """One layer of the query path on the CPU: dequantise the records, attend prefix + suffix
    (over the first n_tok prefix tokens when given: a sample of the layer)."""
    from oracle import pck_oracle as orc
    H_kv, D = W["H_kv"], W["D"]
    Ko = orc.records_to_heads(inp["Krec"][:n_tok], H_kv, D)
    Vo = orc.records_to_heads(inp["Vrec"][:n_tok], H_kv, D)
    Ks, Vs = inp["suf"]
    return orc.prefix_query(inp["Q"], Ko, Vo, None, Ks, Vs)


def _oracle_worker(wid, nw, inq, outq):
    """One host core: builds the layers l with l % nw == wid once, then runs them once per step
    (over the first n_tok prefix tokens of each, when the step is a sample)."""
    mine = [l for l in range(W["layers"]) if l % nw == wid]
    inputs = [oracle_layer_inputs(l) for l in mine]
    outq.put(("ready", wid, 0.0))
    while True:
        msg = inq.get()
        if msg is None:
            return
        n, n_tok = msg
        t0 = time.perf_counter()
        for _ in range(n):
            for inp in inputs:
                oracle_layer(inp, n_tok)
        outq.put(("done", wid, time.perf_counter() - t0))


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        info = open("/proc/cpuinfo").read().splitlines()
        for key in ("model name", "CPU part"):
            for ln in info:
                if ln.lower().startswith(key.lower()):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class OraclePool:
    """The oracle's 16-layer step split over the host cores: one single-threaded process per core
    (at most one per layer), started with `spawn` before any GPU work. run(n) times n steps on
    all workers at once (wall clock from the start signal to the last worker's finish)."""

    def __init__(self):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.nw = max(1, min(os.cpu_count() or 1, W["layers"]))
        self.outq = ctx.Queue()
        self.inqs = [ctx.Queue() for _ in range(self.nw)]
        self.procs = [ctx.Process(target=_oracle_worker, args=(w, self.nw, self.inqs[w], self.outq), daemon=True)
                      for w in range(self.nw)]
        for p in self.procs:
            p.start()
        for _ in range(self.nw):
            self.outq.get()

    def run(self, n, n_tok=None):
        t0 = time.perf_counter()
        for q in self.inqs:
            q.put((n, n_tok))
        for _ in range(self.nw):
            self.outq.get()
        return time.perf_counter() - t0

    def close(self):
        for q in self.inqs:
            q.put(None)
        for p in self.procs:
            p.join(timeout=10)


def time_oracle(budget_s=12.0):
    """cpu_baseline: the oracle's 16-layer step on all host cores for about budget_s seconds."""
    pool = OraclePool()
    try:
        t1 = pool.run(1)                                   # warm-up step, and its duration
        n = max(1, int(budget_s / max(t1, 1e-3)))
        dt = pool.run(n)
    finally:
        pool.close()
    step_s = dt / n
    kv_step = W["layers"] * 2 * W["N"] * REC_BYTES
    return {"value": round(kv_step / step_s / 1e9, 4), "unit": "GB/s", "cores": pool.nw, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"{n} full 16-layer steps of {WORKLOAD} (dequantise records + prefix/suffix attention, fp64 "
                      f"numpy), layers split over {pool.nw} single-threaded processes, {dt:.1f} s",
            "ms_per_step": round(step_s * 1e3, 2)}


def run_reference(args, budget_s=100.0):
    """The CPU oracle as the reference arm: each step is the 16-layer step of the workload, its
    layers split over the host cores; when --steps + --warmup full steps would take more than
    about budget_s, every step attends over the same leading sample of each layer's prefix tokens
    (the bytes counted are those of the sample)."""
    if rank() != 0:
        return
    pool = OraclePool()
    try:
        t_full = pool.run(1)   # one full step: its duration sizes the sample
        n_tok = W["N"]
        total = max(1, args.steps + args.warmup)
        if total * t_full > budget_s:
            n_tok = max(256, int(W["N"] * budget_s / (total * t_full)) // 16 * 16)
        if args.warmup:
            pool.run(args.warmup, n_tok)
        dt = pool.run(args.steps, n_tok)
    finally:
        pool.close()
    kv_step = W["layers"] * 2 * n_tok * REC_BYTES
    val = kv_step * args.steps / dt / 1e9
    what = "full 16-layer steps" if n_tok == W["N"] else \
        f"16-layer steps over the first {n_tok} of the {W['N']} prefix tokens of every layer"
    sample = (f"{args.steps} timed {what} (+{args.warmup} warm-up), layers over {pool.nw} "
              f"single-threaded processes, fp64")
    line = {"metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD, **W, "fmt": "mlx4g32",
                       "step": "the full 16-layer step" if n_tok == W["N"] else
                       f"the 16-layer step over a {n_tok}-token sample of each layer's prefix"},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": pool.nw, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ distributed plumbing

from prefix_cached_kv_gb300.replicas import barrier, max_over_ranks, rank, world   # noqa: E402
from prefix_cached_kv_gb300.replicas import init as dist_init   # noqa: E402
from prefix_cached_kv_gb300.replicas import job_throughput   # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", default="all",
                    help="all | comma list of main,fp16,dims,sparse,prefill,prefill_mlx,cartridge (main = the headline line)")
    ap.add_argument("--profile", default=None,
                    help="fp16 | sparse | quant | warm | prefill | prefill_mlx: one capture-sized run of that row")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.profile:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        from prefix_cached_kv_gb300 import binding
        ctx = binding.Context(torch.cuda.current_device())
        profile_row(args.profile, ctx, torch)
        ctx.close()
        return
    want = {"main", "fp16", "dims", "sparse", "prefill", "prefill_mlx", "cartridge"} if args.rows == "all" \
        else set(args.rows.split(","))
    cpu = time_oracle() if rank() == 0 and "main" in want else None   # before any GPU work
    import torch
    dist_init()
    import __graft_entry__
    __graft_entry__.build()
    from prefix_cached_kv_gb300 import binding
    pk = peaks()
    l2 = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0)) or None
    ctx = binding.Context(torch.cuda.current_device())
    ms_step = steps = clocks = roof = e2e = latency = None
    rows = {}
    if "main" in want:
        ms_step, steps, clocks, roof, e2e, latency = run_main(args, ctx, torch, pk)
        rows["A3_headline_latency_mode"] = latency
        for r in range(ROTATE):
            ctx.drop(f"bench{r}")
    if "fp16" in want:
        rows["A0_A2_fp16_m1"] = row_fp16_m1(ctx, torch, pk)
    if "dims" in want:
        rows["N4_other_head_dims"] = row_dims(ctx, torch, pk)
    if "sparse" in want:
        rows["A6_A7_sparse"] = row_sparse(ctx, torch, pk, l2=l2)
    if "prefill" in want:
        rows["A4_A5_batched_q"] = row_prefill(ctx, torch, pk)
    if "prefill_mlx" in want:
        rows["N3_batched_q_mlx4g32"] = row_prefill(ctx, torch, pk, fmt=1)
    if "cartridge" in want:
        rows["A1_A3_N2_cartridge"] = row_cartridge(ctx, torch, pk)
    ctx.close()
    if rank() != 0:
        return
    if ms_step is None:   # rows only (profiling runs): no headline line
        print(json.dumps({"rows": rows}), flush=True)
        return
    ws = world()
    value = job_throughput(KV_BYTES_STEP, ms_step, ws) / 1e9
    l2_txt = f"{l2 / 2**20:.0f} MiB L2 (device-reported)" if l2 else "L2 size not reported"
    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u4/f16 in, f32 accumulate", "data": "synthetic",
            "config": {"workload": WORKLOAD, **W, "fmt": "mlx4g32",
                       "launch": "16 layers in one batched launch per step, CUDA-graph replayed",
                       "l2": f"rotate {ROTATE} distinct {KV_BYTES_STEP / 1e6:.0f} MB prefix sets "
                             f"({ROTATE * KV_BYTES_STEP / 1e6:.0f} MB vs {l2_txt})",
                       "parallelism": f"replicas x{ws}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": 2 * steps, "rows": rows}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
