"""Benchmark: denoised positions per second of the block-diffusion MoE
denoising step on a Clover-35B-A3B-shaped model (40 MoE layers of 256 experts
top-8 + shared expert, hidden 2,048, SwiGLU 512, untied 248,320-row head,
one block of 32 positions, low-confidence unmask at 0.95).

A step is one pass of the whole hot path over the block: input assembly, 40
MoE sublayers (router, top-8, grouped SwiGLU experts, shared expert,
combine), final norm, head statistics and the unmask rule. Weights are
synthetic (bf16, N(0, 0.02)), resident in HBM; the ~66 GB of weights a step
streams are far larger than L2, so no flush is needed between steps. A block
whose positions are all committed is re-masked before the next step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle on bounded samples of the same
workload (this pool has no other implementation of the method).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_diffusion_moe_gb300 import synth  # noqa: E402

METRIC = "denoised positions/sec per block step (1xGB300); achieved HBM GB/s vs roofline"
UNIT = "positions/s"
D = synth.CLOVER
M = 32
WORKLOAD = "full block denoising step: 40 Clover-shaped MoE layers (256 experts top-8 + shared) + 248,320-row head, " \
           "1 block x 32 positions, unmask threshold 0.95"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _expert_traffic(u_mean, fused, q4=False):
    """DRAM bytes per expert-kernel launch from the committed ncu summary of
    that kernel (bytes per expert x experts per launch), if the summary was
    taken on the current kernel source; else None."""
    name = ("moe_layer_fused_int4_clover_block32.md" if q4 else
            "moe_layer_fused_clover_block32.md" if fused else "moe_layer_standalone_zipf256.md")
    path = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, "block_diffusion_moe_gb300", "csrc", "expert.cu")
    try:
        text = open(path).read()
        sha = text.split("expert.cu sha256:")[1].split()[0]
        per = float(text.split("DRAM bytes per expert (read + write):")[1].split()[0])
        if sha != hashlib.sha256(open(src, "rb").read()).hexdigest() or u_mean is None:
            return None
        return per * (u_mean + 1)
    except Exception:
        return None


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.th = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self

        def rd():
            for line in self.proc.stdout:
                self.rows.append([c.strip() for c in line.split(",")])

        self.th = threading.Thread(target=rd, daemon=True)
        self.th.start()
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.th:
                self.th.join(timeout=2)

    def summary(self):
        rows = [r for r in self.rows if len(r) >= 6]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        return ws, rank, local, dist
    return 1, 0, 0, None


def _barrier(dist):
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()


def _reduce_over_ranks(v: float, dist, op: str) -> float:
    """Max or sum of a per-rank scalar over all ranks (identity with one
    rank). Uses a CPU tensor under gloo and a CUDA tensor under NCCL."""
    if dist is None:
        return v
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def _max_over_ranks(v: float, dist) -> float:
    return _reduce_over_ranks(v, dist, "max")


def _sum_over_ranks(v: float, dist) -> float:
    return _reduce_over_ranks(v, dist, "sum")


def replica_throughput(units_this_rank: float, seconds_this_rank: float, dist) -> float:
    """Whole-job throughput of independent replicas: all ranks' units over the
    slowest rank's time."""
    return _sum_over_ranks(units_this_rank, dist) / _max_over_ranks(seconds_this_rank, dist)


# ---------------------------------------------------------------- CPU oracle


class _LazyBits:
    """Expert-indexed view that copies one expert's bf16 bits to the host on
    first use (the oracle only touches the experts the block routes to)."""

    def __init__(self, t):
        self.t, self.c = t, {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.c:
            self.c[e] = synth.bf16_bits(self.t[e])
        return self.c[e]


def cpu_baseline(layers=None, n_layers: int = 40, head_rows: int = 24832, seed: int = 0):
    """Oracle timing on the host cores: n_layers MoE layers of the
    32-position block plus head_rows rows of the head, scaled to one full
    step (40 layers, 248,320 rows). `layers` are resident synth layers (any
    device); without them, n_layers layers are drawn on the CPU."""
    import oracle as O

    if layers is None:
        layers = [synth.make_layer(D, seed, l, "cpu") for l in range(n_layers)]
    layers = layers[:n_layers]
    head = synth.normal((head_rows, D.hidden), synth.WEIGHT_STD, 424242, "cpu")
    ctx = synth.make_ctx(D, M, seed, "cpu").numpy()
    mask_row = synth.normal((1, D.hidden), 1.0, 434343, "cpu")
    x = O.embed(np.zeros(M, dtype=np.int32), synth.bf16_bits(mask_row), ctx)
    tl = 0.0
    for L in layers:
        lay = {"router_w": synth.bf16_bits(L.router_w), "gate_up": _LazyBits(L.gate_up),
               "down": _LazyBits(L.down), "sh_gate_up": synth.bf16_bits(L.sh_gate_up),
               "sh_down": synth.bf16_bits(L.sh_down), "router_bias": None}
        idx = O.route(O.round_to_bf16(O.rms_norm(x, D.rms_eps)), lay["router_w"], D.top_k)[2]
        for e in np.unique(idx):          # host copies happen outside the timed part
            lay["gate_up"][e], lay["down"][e]
        a = time.perf_counter()
        x = O.moe_layer(x, lay, D.top_k, D.rms_eps)["x_out"]
        tl += time.perf_counter() - a
    a = time.perf_counter()
    z = O.head_logits(x, synth.bf16_bits(head), D.rms_eps)
    O.head_stats(z, 0)
    th = time.perf_counter() - a
    per_layer = tl / len(layers)
    head_full = th * (D.vocab / head_rows)
    desc = (f"oracle (numpy float64, BLAS threads = host cores) on {len(layers)} MoE layers of the 32-position "
            f"block ({tl:.1f} s) and {head_rows} of {D.vocab} head rows ({th:.1f} s), scaled to 40 layers + "
            f"full head")
    return per_layer, head_full, desc, os.cpu_count()


# ------------------------------------------------------------------- arms


def run_reference(args):
    ws, rank, local, dist = _dist()
    if rank != 0:
        return
    per = []
    desc = ""
    cores = os.cpu_count()
    ref_layers = [synth.make_layer(D, 0, 0, "cpu")]
    for i in range(args.warmup + args.steps):
        pl, hf, desc, cores = cpu_baseline(layers=ref_layers, n_layers=1, head_rows=4096, seed=i)
        if i >= args.warmup:
            per.append(pl * D.n_layers + hf)
    sec = float(np.mean(per))
    value = M / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": M, "seq_len": M, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


WORKLOADS = {
    "step": WORKLOAD,
    "layer": "one Clover-shaped MoE layer (256 experts top-8 + shared, hidden 2,048, SwiGLU 512) on a "
             "32-position block, uniform routing",
    "head": "LM head + low-confidence unmask: 32 positions x hidden 2,048 into the untied 248,320-row head",
    "accept": "verify-pass head + self-speculative accept test (exact rule): one block of 32 drafts (33 rows x hidden "
              "2,048) into the untied 248,320-row head",
    "zipf": "batched and skewed routing: 8 blocks x 32 positions (256 tokens) through 40 Clover-shaped MoE "
            "layers + head, router biased to Zipf(1.2) expert popularity",
    "coreset": "full block denoising step as 'step' with the block coreset expert selection (top_p 0.9) in every "
               "MoE layer",
    "int4": "full block denoising step as 'step' with every expert's weights in the 4-bit format (4-bit codes, one "
            "bf16 scale per 64 weights: 1,671,168 B per expert instead of 6,291,456 B)",
    "zipf_layer": "one Clover-shaped MoE layer on 8 blocks x 32 positions (256 tokens), router biased to Zipf(1.2) "
                  "expert popularity (the standalone routing and expert kernels)",
    "int4_layer": "one Clover-shaped MoE layer on a 32-position block with every expert's weights in the 4-bit "
                  "format (the size ncu captures of the low-bit kernel use)",
}
CORESET_TOP_P = 0.9


def run_ours(args):
    from block_diffusion_moe_gb300 import clover

    ws_n, rank, local, dist = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    clover.lib()
    seed = 1000 + rank
    kind = args.workload
    n_pos = 256 if kind in ("zipf", "zipf_layer") else M
    n_layers = {"step": D.n_layers, "zipf": D.n_layers, "coreset": D.n_layers, "int4": D.n_layers, "layer": 1,
                "zipf_layer": 1, "int4_layer": 1,
                "head": 0, "accept": 0}[kind]
    head_like = kind in ("head", "accept")
    if kind == "accept":
        n_pos = M + 1
    one_layer = kind in ("layer", "zipf_layer", "int4_layer")
    q4 = kind in ("int4", "int4_layer")
    full = kind in ("step", "zipf", "coreset", "int4")
    top_p = CORESET_TOP_P if kind == "coreset" else 0.0
    zipf = 1.2 if kind in ("zipf", "zipf_layer") else None
    layers = [synth.make_layer(D, seed, l, dev, zipf_s=zipf) for l in range(n_layers)]
    if q4:
        # the library's own quantizer; the bf16 expert weights are dropped after
        layers = [clover.quantize_layer_q4(L) for L in layers]
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    head_w = synth.make_head(D, seed, dev) if not one_layer else None
    embed = synth.make_embed(D, seed, dev) if full else None
    model = clover.Model(D, layers, embed, head_w, coreset_top_p=top_p) if full else None
    ctx = synth.make_ctx(D, n_pos, seed, dev)
    tokens, masked = synth.masked_block(D, n_pos, dev)
    stream = torch.cuda.current_stream(dev)
    x_fixed = synth.make_x(D, n_pos, seed, dev)
    x_out = torch.empty_like(x_fixed)
    if full:
        ws = clover.workspace(clover.denoise_workspace_bytes(D, n_pos), dev)
    elif one_layer:
        ws = clover.workspace(clover.moe_workspace_bytes(D, n_pos), dev)
    elif kind == "accept":
        ws = clover.workspace(clover.accept_workspace_bytes(D, n_pos), dev)
    else:
        ws = clover.workspace(clover.head_workspace_bytes(D, n_pos), dev)
    draft = acc_out = None
    if kind == "accept":
        # drafts: the head's own argmax with every fourth row replaced by a
        # seeded random id (a stand-in for the preview pass's candidates)
        acc_out = clover.lmhead_accept(D, head_w, x_fixed, torch.zeros(n_pos, dtype=torch.int32, device=dev), n_pos,
                                       ws=ws)
        g = torch.Generator(device="cpu").manual_seed(seed)
        draft = acc_out["argmax"].clone()
        draft[3::4] = torch.randint(0, D.vocab, (len(range(3, n_pos, 4)),), generator=g).to(torch.int32).to(dev)
        draft[-1] = -1

    def reset():
        tokens.fill_(D.mask_id)
        masked.fill_(1)

    steps_in_block = [0]

    def step():
        if full:
            if steps_in_block[0] == M:
                reset()
                steps_in_block[0] = 0
            clover.denoise_step(model, ctx, tokens, masked, block=M, ws=ws)
            steps_in_block[0] += 1
        elif one_layer:
            clover.moe_block_step(D, layers[0], x_fixed, x_out=x_out, ws=ws, with_topk=False)
        else:
            if kind == "accept":
                clover.lmhead_accept(D, head_w, x_fixed, draft, n_pos, clover.ACCEPT_EXACT, ws=ws, out=acc_out)
            else:
                clover.lmhead_unmask(D, head_w, x_fixed, tokens, masked, block=M, ws=ws)

    for _ in range(args.warmup):
        step()
    reset()
    steps_in_block[0] = 0
    torch.cuda.synchronize()
    clover.workspace_status(ws)

    # ---- timed region: device time of K steps; per-launch events around the
    # dominant kernel (the expert kernel, or the whole head call)
    per_step_launches = n_layers if not head_like else 1
    n_ev = args.steps * per_step_launches
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for e in ev_b + ev_e:          # torch creates the CUDA event on first record
        e.record(stream)
    torch.cuda.synchronize()
    arr_b = (clover.ctypes.c_void_p * n_ev)(*[e.cuda_event for e in ev_b])
    arr_e = (clover.ctypes.c_void_p * n_ev)(*[e.cuda_event for e in ev_e])
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(dist)
    start2, end2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        # (1) the headline: K steps with nothing between the kernels
        start.record(stream)
        for i in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        # (2) the same K steps again, with events around every launch of the
        # dominant kernel (they sit between kernels, so this pass runs a little
        # slower; it only feeds the roofline figure)
        reset()
        steps_in_block[0] = 0
        if not head_like:
            clover.lib().clover_profile_expert_events(arr_b, arr_e, n_ev)
        start2.record(stream)
        for i in range(args.steps):
            if head_like:
                ev_b[i].record(stream)
            step()
            if head_like:
                ev_e[i].record(stream)
        end2.record(stream)
        torch.cuda.synchronize()
        recorded = clover.lib().clover_profile_expert_events(None, None, 0) if not head_like else n_ev
    _barrier(dist)
    clover.workspace_status(ws)
    ms = start.elapsed_time(end)
    ms_instr = start2.elapsed_time(end2)
    assert recorded == n_ev, (recorded, n_ev)
    durs = [b.elapsed_time(e) for b, e in zip(ev_b, ev_e)]

    # ---- algorithmic bytes: replay the same steps layer by layer (the kernels
    # are deterministic) and count the experts each launch touched.
    # per expert: bf16 weights, or 4-bit codes + one bf16 scale per 64 weights
    ebytes = D.expert_bytes if not q4 else D.expert_params // 2 + D.expert_params // 64 * 2
    u_per_launch = []
    if head_like:
        alg = [D.head_bytes] * n_ev
    else:
        reset()
        x = torch.empty((n_pos, D.hidden), dtype=torch.float32, device=dev)
        moe_ws = clover.workspace(clover.moe_workspace_bytes(D, n_pos), dev)
        head_ws = clover.workspace(clover.head_workspace_bytes(D, n_pos), dev)
        for s_ in range(args.steps):
            if one_layer:
                _, idx, _ = clover.moe_block_step(D, layers[0], x_fixed, x_out=x, ws=moe_ws)
                u_per_launch.append(int(torch.unique(idx).numel()))
                continue
            if s_ > 0 and s_ % M == 0:
                reset()
            x.copy_(model.embed[tokens.long()].float() + ctx)
            for L in layers:
                x, idx, _ = clover.moe_block_step(D, L, x, x_out=x, ws=moe_ws, coreset_top_p=top_p)
                u_per_launch.append(int(torch.unique(idx).numel()))
            clover.lmhead_unmask(D, head_w, x, tokens, masked, block=M, ws=head_ws)
        torch.cuda.synchronize()
        alg = [(u + 1) * ebytes for u in u_per_launch]
    achieved = sum(alg) / (sum(durs) * 1e-3) / 1e9          # GB/s
    peak, peak_kind = _peaks()
    u_mean = float(np.mean(u_per_launch)) if u_per_launch else None
    # (for the head workloads alg already is the head's bytes)
    step_bytes = sum(alg) / args.steps + n_layers * D.router_bytes + (D.head_bytes if full else 0)
    share = sum(durs) / ms_instr

    # ---- end to end through the C ABI with host buffers
    h_tokens = torch.empty(n_pos, dtype=torch.int32).pin_memory()
    h_masked = torch.empty(n_pos, dtype=torch.uint8).pin_memory()
    h_in = (x_fixed if one_layer or head_like else ctx).cpu().pin_memory()
    d_in = x_fixed if one_layer or head_like else ctx
    o_tokens = torch.empty(n_pos, dtype=torch.int32).pin_memory()
    o_masked = torch.empty(n_pos, dtype=torch.uint8).pin_memory()
    o_x = torch.empty((n_pos, D.hidden), dtype=torch.float32).pin_memory()
    h_draft = draft.cpu().pin_memory() if kind == "accept" else None
    o_len = torch.empty(1, dtype=torch.int32).pin_memory()
    def e2e_step(s_):
        if full and s_ > 0 and s_ % M == 0:
            h_tokens.fill_(D.mask_id)
            h_masked.fill_(1)
        d_in.copy_(h_in, non_blocking=True)
        if kind == "accept":
            draft.copy_(h_draft, non_blocking=True)
        elif not one_layer:
            tokens.copy_(h_tokens, non_blocking=True)
            masked.copy_(h_masked, non_blocking=True)
        if full:
            clover.denoise_step(model, ctx, tokens, masked, block=M, ws=ws)
        else:
            step()
        if one_layer:
            o_x.copy_(x_out, non_blocking=True)
        elif kind == "accept":
            o_tokens.copy_(acc_out["tokens"], non_blocking=True)
            o_len.copy_(acc_out["accept_len"][:1], non_blocking=True)
        else:
            o_tokens.copy_(tokens, non_blocking=True)
            o_masked.copy_(masked, non_blocking=True)
        torch.cuda.synchronize()
        if full:
            h_tokens.copy_(o_tokens)
            h_masked.copy_(o_masked)

    # one untimed pass first (first-use costs of the pinned buffers and copies)
    h_tokens.fill_(D.mask_id)
    h_masked.fill_(1)
    e2e_step(0)
    h_tokens.fill_(D.mask_id)
    h_masked.fill_(1)
    steps_in_block[0] = 0
    _barrier(dist)
    t0 = time.perf_counter()
    for s_ in range(args.steps):
        e2e_step(s_)
    e2e_s = time.perf_counter() - t0
    if one_layer:
        h2d, d2h = n_pos * D.hidden * 4, n_pos * D.hidden * 4
    elif kind == "accept":
        h2d, d2h = n_pos * D.hidden * 4 + n_pos * 4, n_pos * 4 + 4
    else:
        h2d = n_pos * 4 + n_pos + n_pos * D.hidden * 4
        d2h = n_pos * 4 + n_pos

    # collectives: every rank takes part before rank 0 alone reports
    value = replica_throughput(n_pos * args.steps, ms * 1e-3, dist)
    e2e_value = replica_throughput(n_pos * args.steps, e2e_s, dist)
    ms_max = _max_over_ranks(ms, dist)
    if rank != 0:
        return
    csum = clk.summary()
    # <= 32 positions: one fused launch per layer; more: route, experts (with the permutation), combine
    per_layer = 1 if n_pos <= 32 else 3
    launches_per_step = {"step": 1 + per_layer * n_layers + 2, "zipf": 1 + per_layer * n_layers + 2,
                         "coreset": 1 + per_layer * n_layers + 2, "int4": 1 + per_layer * n_layers + 2, "layer": per_layer, "zipf_layer": per_layer,
                         "int4_layer": per_layer,
                         "head": 2, "accept": 2}[kind]
    roof_kernel = ("k_head + k_rmsnorm (head statistics and unmask)" if kind == "head"
                   else "k_head<accept> + k_rmsnorm (head statistics, entropy and the accept test)"
                   if kind == "accept"
                   else "k_layer (routing + grouped SwiGLU experts + combine, one launch per MoE layer)"
                   if n_pos <= 32 else "k_expert (grouped SwiGLU experts + combine, one launch per MoE layer)")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded random-init bf16 weights of the Clover shapes)",
        "config": {"workload": WORKLOADS[kind], "global_batch": n_pos * ws_n, "seq_len": M,
                   "parallelism": "replicas" if ws_n > 1 else "single",
                   "l2": "inputs larger than L2 (every step streams >= 1 GB of weights)",
                   "mean_unique_experts_per_layer": u_mean,
                   "algorithmic_bytes_per_step": step_bytes,
                   "step_hbm_gbs": step_bytes / (ms_max / args.steps * 1e-3) / 1e9,
                   "step_roofline_frac": step_bytes / (ms_max / args.steps * 1e-3) / 1e9 / peak},
        "roofline": {"kernel": roof_kernel, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": _expert_traffic(u_mean, n_pos <= 32, q4) if not head_like else None,
                     "launches": len(durs),
                     "mean_launch_us": float(np.mean(durs)) * 1e3, "share_of_step": share,
                     "ms_per_step_with_events": ms_instr / args.steps},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": csum,
    }
    if not args.no_cpu_baseline and kind in ("step", "layer"):
        pl, hf, desc, cores = cpu_baseline(layers=layers)
        sec = pl * D.n_layers + hf if kind == "step" else pl
        line["cpu_baseline"] = {"value": M / sec, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="step", choices=sorted(WORKLOADS),
                    help="step (default, the headline): full 40-layer block step; layer / head / zipf: the other "
                         "configurations")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
