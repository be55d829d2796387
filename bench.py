"""Benchmark: denoised positions per second of the block-diffusion MoE
denoising step on a Clover-35B-A3B-shaped model (40 MoE layers of 256 experts
top-8 + shared expert, hidden 2,048, SwiGLU 512, untied 248,320-row head,
one block of 32 positions, low-confidence unmask at 0.95).

A step is one pass of the whole hot path over the block: input assembly, 40
MoE sublayers (router, top-8, grouped SwiGLU experts, shared expert,
combine), final norm, head statistics and the unmask rule. Weights are
synthetic (bf16, N(0, 0.02)), resident in HBM; the ~66 GB of weights a step
streams are far larger than L2, so no flush is needed between steps.

The cost of a step depends on where it falls in its block: early steps have
more masked slots, which share the mask token's embedding and so touch fewer
distinct experts. The K timed steps are therefore taken from K copies of the
block at evenly spaced points of the denoising loop (copy i enters the timed
region with floor(32 i / K) of its slots committed), so that they carry the
mix of a whole block. The end-to-end figure runs whole blocks through
clover_denoise_block, the loop entry point.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the CPU oracle (this pool has no other implementation
of the method) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

if "--oracle-1core" in sys.argv:
    # the single-thread oracle figure runs in a child process whose BLAS is
    # limited to one thread before numpy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_diffusion_moe_gb300 import synth  # noqa: E402

METRIC = "denoised positions/sec per block step (1xGB300); achieved HBM GB/s vs roofline"
UNIT = "positions/s"
D = synth.CLOVER
M = 32
WORKLOAD = "full block denoising step: 40 Clover-shaped MoE layers (256 experts top-8 + shared) + 248,320-row head, " \
           "1 block x 32 positions, unmask threshold 0.95"

WORKLOADS = {
    "step": WORKLOAD,
    "layer": "one Clover-shaped MoE layer (256 experts top-8 + shared, hidden 2,048, SwiGLU 512) on a "
             "32-position block, uniform routing",
    "head": "LM head + low-confidence unmask: 32 positions x hidden 2,048 into the untied 248,320-row head",
    "accept": "verify-pass head + self-speculative accept test (exact rule): one block of 32 drafts (33 rows x hidden "
              "2,048) into the untied 248,320-row head",
    "zipf": "batched and skewed routing: 8 blocks x 32 positions (256 tokens) through 40 Clover-shaped MoE "
            "layers + head, router biased to Zipf(1.2) expert popularity",
    "zipf512": "batching beyond 8 blocks: 16 blocks x 32 positions (512 tokens) through 40 Clover-shaped MoE "
               "layers + head, router biased to Zipf(1.2) expert popularity (hot experts take more than 256 tokens)",
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


class Spec:
    """What a workload runs: token count, layers, and which entry point."""

    def __init__(self, kind: str):
        self.kind = kind
        self.n_pos = {"zipf": 256, "zipf_layer": 256, "zipf512": 512, "accept": M + 1}.get(kind, M)
        self.n_layers = {"step": D.n_layers, "zipf": D.n_layers, "zipf512": D.n_layers, "coreset": D.n_layers,
                         "int4": D.n_layers,
                         "layer": 1, "zipf_layer": 1, "int4_layer": 1, "head": 0, "accept": 0}[kind]
        self.head_like = kind in ("head", "accept")
        self.one_layer = kind in ("layer", "zipf_layer", "int4_layer")
        self.q4 = kind in ("int4", "int4_layer")
        self.full = kind in ("step", "zipf", "zipf512", "coreset", "int4")
        self.top_p = CORESET_TOP_P if kind == "coreset" else 0.0
        self.zipf = 1.2 if kind in ("zipf", "zipf_layer", "zipf512") else None


def base_config(kind: str, n_gpus: int) -> dict:
    """The workload description both arms print (identical for the same
    workload and GPU count)."""
    sp = Spec(kind)
    return {"workload": WORKLOADS[kind], "global_batch": sp.n_pos * n_gpus, "seq_len": M,
            "parallelism": "replicas" if n_gpus > 1 else "single",
            "l2": "inputs larger than L2 (every step streams >= 1 GB of weights)"}


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


def block_phases(k: int, block: int = M) -> list:
    """Evenly spaced points of a block's denoising loop for k timed steps:
    step i starts with floor(block * i / k) slots committed."""
    return [(block * i) // k for i in range(k)]


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


class _DrawnExperts:
    """Expert-indexed bf16 bits drawn on the host on first use
    (synth.make_expert); part 0 = gate_up, 1 = down. The pair is drawn once
    and shared by both views."""

    def __init__(self, seed, layer, cache, part):
        self.seed, self.layer, self.cache, self.part = seed, layer, cache, part

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            gu, dn = synth.make_expert(D, self.seed, self.layer, e, "cpu")
            self.cache[e] = (synth.bf16_bits(gu), synth.bf16_bits(dn))
        return self.cache[e][self.part]


def host_layer(seed: int, layer: int, zipf_s=None) -> dict:
    """One layer in the oracle's input format, drawn on the host: the router
    and shared expert at once, routed experts when first touched."""
    cache = {}
    return {"router_w": synth.bf16_bits(synth.make_router(D, seed, layer, "cpu")),
            "gate_up": _DrawnExperts(seed, layer, cache, 0), "down": _DrawnExperts(seed, layer, cache, 1),
            "sh_gate_up": synth.bf16_bits(synth.normal((2 * D.d_ff, D.hidden), synth.WEIGHT_STD,
                                                       synth._seed(seed, layer, "sh_gate_up"), "cpu")),
            "sh_down": synth.bf16_bits(synth.normal((D.hidden, D.d_ff), synth.WEIGHT_STD,
                                                    synth._seed(seed, layer, "sh_down"), "cpu")),
            "router_bias": None if zipf_s is None
            else synth.zipf_router_bias(D, seed, layer, zipf_s, "cpu").numpy().astype(np.float32)}


def device_layer(L) -> dict:
    """A device-resident synth layer in the oracle's input format (experts
    copied to the host when first touched)."""
    return {"router_w": synth.bf16_bits(L.router_w), "gate_up": _LazyBits(L.gate_up), "down": _LazyBits(L.down),
            "sh_gate_up": synth.bf16_bits(L.sh_gate_up), "sh_down": synth.bf16_bits(L.sh_down),
            "router_bias": None if L.router_bias is None else L.router_bias.cpu().numpy().astype(np.float32)}


def _block_input(seed: int, n_pos: int = M):
    """The oracle's input for a freshly opened block: the mask token's
    embedding (one row drawn on the host) plus the context term."""
    import oracle as O
    ctx = synth.make_ctx(D, n_pos, seed, "cpu").numpy()
    mask_row = synth.normal((1, D.hidden), 1.0, 434343, "cpu")
    return O.embed(np.zeros(n_pos, dtype=np.int32), synth.bf16_bits(mask_row), ctx)


def time_oracle(layers, x, head_rows: int):
    """Wall time of the oracle on the block x: every layer of `layers`
    (oracle-format dicts, run in order), then head statistics over head_rows
    rows of a head. The experts a layer routes to are copied or drawn before
    its timed part. Returns (seconds per layer list, head seconds, x out)."""
    import oracle as O
    t_layers = []
    for lay in layers:
        idx = O.route(O.round_to_bf16(O.rms_norm(x, D.rms_eps)), lay["router_w"], D.top_k,
                      lay.get("router_bias"))[2]
        for e in np.unique(idx):
            lay["gate_up"][e], lay["down"][e]
        a = time.perf_counter()
        x = O.moe_layer(x, lay, D.top_k, D.rms_eps)["x_out"]
        t_layers.append(time.perf_counter() - a)
    t_head = 0.0
    if head_rows > 0:
        head = _HEAD_ROWS.get(head_rows)
        if head is None:
            head = _HEAD_ROWS[head_rows] = synth.bf16_bits(synth.normal((head_rows, D.hidden), synth.WEIGHT_STD,
                                                                        424242, "cpu"))
        a = time.perf_counter()
        z = O.head_logits(x, head, D.rms_eps)
        O.head_stats(z, 0)
        t_head = time.perf_counter() - a
    return t_layers, t_head, x


_HEAD_ROWS = {}


def oracle_1core(kind: str) -> dict:
    """The single-thread oracle figure: a child process with its BLAS limited
    to one thread times one layer (drawn on the host) and a hundredth of the
    head rows, scaled to the workload's unit."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-1core", "--workload", kind]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=240)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal: the all-core figure stands alone
        return {"error": f"single-thread oracle run failed: {type(e).__name__}"}


def _oracle_1core_child(kind: str):
    sp = Spec(kind)
    x = _block_input(7)
    t_layers, t_head, _ = time_oracle([host_layer(7, 0)] if sp.n_layers else [], x,
                                      D.vocab // 100 if (sp.full or sp.head_like) else 0)
    per_layer = t_layers[0] if t_layers else 0.0
    head_full = t_head * 100
    sec = per_layer * sp.n_layers + (head_full if (sp.full or sp.head_like) else 0.0)
    print(json.dumps({"value": M / sec, "unit": UNIT, "cores": 1,
                      "sample": f"oracle with one BLAS thread on 1 MoE layer ({per_layer:.2f} s) and "
                                f"{D.vocab // 100} head rows ({t_head:.2f} s), scaled to the workload"}))


def cpu_baseline(sp: Spec, layers) -> dict:
    """The oracle on all host cores on a bounded sample of the workload, and
    the same on one core (child process)."""
    x = _block_input(0)
    if sp.full:
        # all 40 layers of the step (device weights copied when touched) and a
        # tenth of the head rows
        t_layers, t_head, _ = time_oracle([device_layer(L) for L in layers], x, D.vocab // 10)
        sec = sum(t_layers) + t_head * 10
        desc = (f"oracle (numpy float64, BLAS threads = host cores) on the {len(t_layers)} MoE layers of the "
                f"32-position block ({sum(t_layers):.1f} s) and {D.vocab // 10} of {D.vocab} head rows "
                f"({t_head:.1f} s), head scaled to all rows")
    elif sp.one_layer:
        t_layers, _, _ = time_oracle([device_layer(layers[0])], x, 0)
        sec = t_layers[0]
        desc = f"oracle (numpy float64, BLAS threads = host cores) on one MoE layer of 32 positions ({sec:.2f} s)"
    else:
        _, t_head, _ = time_oracle([], x, D.vocab // 10)
        sec = t_head * 10
        desc = (f"oracle (numpy float64, BLAS threads = host cores) head statistics of 32 positions over "
                f"{D.vocab // 10} of {D.vocab} head rows ({t_head:.1f} s), scaled to all rows")
    out = {"value": M / sec, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
           "workload_positions": M}
    one = oracle_1core(sp.kind)
    out["one_core"] = one
    return out


# ------------------------------------------------------------------- arms


def run_reference(args):
    """The oracle as the reference arm: each timed step is a bounded sample
    of the workload (a stated fraction of one step's work), timed on the host
    cores; value = positions of a step x that fraction / sample seconds."""
    ws, rank, local, dist = _dist()
    if rank != 0:
        return
    sp = Spec(args.workload)
    if sp.full:
        n_lay, rows, frac = 4, D.vocab // 10, 0.1      # 4 of 40 layers and a tenth of the head rows
    elif sp.one_layer:
        n_lay, rows, frac = 1, 0, 1.0
    else:
        n_lay, rows, frac = 0, D.vocab // 10, 0.1
    layers = [host_layer(0, l, sp.zipf) for l in range(n_lay)]
    x0 = _block_input(0, M)
    secs = []
    for i in range(args.warmup + args.steps):
        tl, th, _ = time_oracle(layers, x0, rows)
        if i >= args.warmup:
            secs.append(sum(tl) + th)
    sec = float(np.mean(secs))
    value = M * frac / sec
    desc = (f"oracle (numpy float64, BLAS threads = host cores); each step times {n_lay} MoE layer(s) of the "
            f"32-position block and {rows} of {D.vocab} head rows = {frac:g} of one step's work; value = 32 x "
            f"{frac:g} positions / seconds per timed sample (extrapolated from the sample)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": base_config(args.workload, 1),
            "step_fraction": frac, "extrapolated": True,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if sp.zipf is not None:
        line["note"] = "one block of 32 of the 8 (the oracle's cost is linear in the positions)"
    print(json.dumps(line), flush=True)


def run_ours(args):
    from block_diffusion_moe_gb300 import clover

    ws_n, rank, local, dist = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    clover.lib()
    seed = 1000 + rank
    sp = Spec(args.workload)
    kind, n_pos, n_layers = sp.kind, sp.n_pos, sp.n_layers
    K, W = args.steps, args.warmup
    layers = [synth.make_layer(D, seed, l, dev, zipf_s=sp.zipf) for l in range(n_layers)]
    if sp.q4:
        # the library's own quantizer; the bf16 expert weights are dropped after
        layers = [clover.quantize_layer_q4(L) for L in layers]
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    head_w = synth.make_head(D, seed, dev) if not sp.one_layer else None
    embed = synth.make_embed(D, seed, dev) if sp.full else None
    model = clover.Model(D, layers, embed, head_w, coreset_top_p=sp.top_p) if sp.full else None
    ctx = synth.make_ctx(D, n_pos, seed, dev)
    stream = torch.cuda.current_stream(dev)
    x_fixed = synth.make_x(D, n_pos, seed, dev)
    x_out = torch.empty_like(x_fixed)
    if sp.full:
        ws = clover.workspace(clover.denoise_workspace_bytes(D, n_pos), dev)
    elif sp.one_layer:
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
    tokens, masked = synth.masked_block(D, n_pos, dev)
    head_out = (clover.lmhead_unmask(D, head_w, x_fixed, tokens.clone(), masked.clone(), block=M, ws=ws)
                if kind == "head" else None)

    # ---- block states for the full step: K copies of the block at evenly
    # spaced points of its loop, prepared by one walk through a block
    phases = block_phases(K) if sp.full else []
    init_tok, init_msk = [None] * K, [None] * K
    if sp.full:
        for i in range(W):                       # warm-up steps on a block of their own
            if i % M == 0:
                tokens.fill_(D.mask_id)
                masked.fill_(1)
            clover.denoise_step(model, ctx, tokens, masked, block=M, ws=ws)
        tokens.fill_(D.mask_id)
        masked.fill_(1)
        for ph in range(max(phases) + 1):
            for i, p in enumerate(phases):
                if p == ph:
                    init_tok[i], init_msk[i] = tokens.clone(), masked.clone()
            if ph < max(phases):
                clover.denoise_step(model, ctx, tokens, masked, block=M, ws=ws)
        tok = [t.clone() for t in init_tok]
        msk = [m.clone() for m in init_msk]
    torch.cuda.synchronize()

    def restore():
        for i in range(K):
            tok[i].copy_(init_tok[i])
            msk[i].copy_(init_msk[i])

    def step(i):
        if sp.full:
            clover.denoise_step(model, ctx, tok[i], msk[i], block=M, ws=ws)
        elif sp.one_layer:
            clover.moe_block_step(D, layers[0], x_fixed, x_out=x_out, ws=ws, with_topk=False)
        elif kind == "accept":
            clover.lmhead_accept(D, head_w, x_fixed, draft, n_pos, clover.ACCEPT_EXACT, ws=ws, out=acc_out)
        else:
            clover.lmhead_unmask(D, head_w, x_fixed, tokens, masked, block=M, ws=ws, out=head_out)

    if not sp.full:
        for _ in range(W):
            step(0)
    torch.cuda.synchronize()
    clover.workspace_status(ws)

    # ---- timed region: device time of K steps; then the same K steps again
    # with events around every launch of the dominant kernel
    per_step_launches = n_layers if not sp.head_like else 1
    n_ev = K * per_step_launches
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    for e in ev_b + ev_e:          # torch creates the CUDA event on first record
        e.record(stream)
    torch.cuda.synchronize()
    arr_b = (clover.ctypes.c_void_p * n_ev)(*[e.cuda_event for e in ev_b])
    arr_e = (clover.ctypes.c_void_p * n_ev)(*[e.cuda_event for e in ev_e])
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start2, end2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sp.full:
        restore()
    _barrier(dist)
    with Clocks(local) as clk:
        # (1) the headline: K steps with nothing between the kernels
        start.record(stream)
        for i in range(K):
            step(i)
        end.record(stream)
        torch.cuda.synchronize()
        committed = (sum(int(init_msk[i].sum()) - int(msk[i].sum()) for i in range(K)) if sp.full else 0)
        # (2) the same K steps again, with events around every launch of the
        # dominant kernel (events between launches keep each launch from
        # overlapping its predecessor's tail, so these per-launch times are an
        # upper bound; they only feed the roofline figure)
        if sp.full:
            restore()
        if not sp.head_like:
            clover.lib().clover_profile_expert_events(arr_b, arr_e, n_ev)
        start2.record(stream)
        for i in range(K):
            if sp.head_like:
                ev_b[i].record(stream)
            step(i)
            if sp.head_like:
                ev_e[i].record(stream)
        end2.record(stream)
        torch.cuda.synchronize()
        recorded = clover.lib().clover_profile_expert_events(None, None, 0) if not sp.head_like else n_ev
    _barrier(dist)
    clover.workspace_status(ws)
    ms = start.elapsed_time(end)
    ms_instr = start2.elapsed_time(end2)
    assert recorded == n_ev, (recorded, n_ev)
    durs = [b.elapsed_time(e) for b, e in zip(ev_b, ev_e)]

    # ---- algorithmic bytes: replay the same steps layer by layer (the kernels
    # are deterministic) and count the experts each launch touched.
    # per expert: bf16 weights, or 4-bit codes + one bf16 scale per 64 weights
    ebytes = D.expert_bytes if not sp.q4 else D.expert_params // 2 + D.expert_params // 64 * 2
    u_per_launch = []
    if sp.head_like:
        alg = [D.head_bytes] * n_ev
    else:
        x = torch.empty((n_pos, D.hidden), dtype=torch.float32, device=dev)
        moe_ws = clover.workspace(clover.moe_workspace_bytes(D, n_pos), dev)
        head_ws = clover.workspace(clover.head_workspace_bytes(D, n_pos), dev)
        for s_ in range(K):
            if sp.one_layer:
                _, idx, _ = clover.moe_block_step(D, layers[0], x_fixed, x_out=x, ws=moe_ws)
                u_per_launch.append(int(torch.unique(idx).numel()))
                continue
            x.copy_(model.embed[init_tok[s_].long()].float() + ctx)
            for L in layers:
                x, idx, _ = clover.moe_block_step(D, L, x, x_out=x, ws=moe_ws, coreset_top_p=sp.top_p)
                u_per_launch.append(int(torch.unique(idx).numel()))
        torch.cuda.synchronize()
        del head_ws
        alg = [(u + 1) * ebytes for u in u_per_launch]
    achieved = sum(alg) / (sum(durs) * 1e-3) / 1e9          # GB/s
    peak, peak_kind = _peaks()
    u_mean = float(np.mean(u_per_launch)) if u_per_launch else None
    # (for the head workloads alg already is the head's bytes)
    step_bytes = sum(alg) / K + n_layers * D.router_bytes + (D.head_bytes if sp.full else 0)
    share = sum(durs) / ms_instr

    # ---- end to end through the C ABI with host buffers
    if sp.full:
        # whole blocks through clover_denoise_block (the loop entry point: one
        # host read of the masked count per step), the block's inputs copied
        # from pinned host memory and its tokens read back
        n_blocks = max(1, math.ceil(K / M))
        h_ctx = ctx.cpu().pin_memory()
        h_tokens = torch.full((n_pos,), D.mask_id, dtype=torch.int32).pin_memory()
        h_masked = torch.ones(n_pos, dtype=torch.uint8).pin_memory()
        o_tokens = torch.empty(n_pos, dtype=torch.int32).pin_memory()
        o_masked = torch.empty(n_pos, dtype=torch.uint8).pin_memory()
        e_tok, e_msk = torch.empty_like(tokens), torch.empty_like(masked)

        def e2e_block():
            ctx.copy_(h_ctx, non_blocking=True)
            e_tok.copy_(h_tokens, non_blocking=True)
            e_msk.copy_(h_masked, non_blocking=True)
            n = clover.denoise_block(model, ctx, e_tok, e_msk, block=M, max_steps=M, ws=ws)
            o_tokens.copy_(e_tok, non_blocking=True)
            o_masked.copy_(e_msk, non_blocking=True)
            torch.cuda.synchronize()
            assert int(o_masked.sum()) == 0
            return n

        e2e_block()                              # untimed: first use of the buffers
        _barrier(dist)
        t0 = time.perf_counter()
        e2e_steps = sum(e2e_block() for _ in range(n_blocks))
        e2e_s = time.perf_counter() - t0
        e2e_units = n_pos * e2e_steps
        h2d = (ctx.numel() * 4 + n_pos * 4 + n_pos) * n_blocks / e2e_steps
        # per block: the initial mask read, 12 bytes of status per step, tokens and mask back
        d2h = (n_pos + 12 * e2e_steps + n_pos * 5 * n_blocks) / e2e_steps
        e2e_extra = {"blocks": n_blocks, "steps": e2e_steps, "entry_point": "clover_denoise_block",
                     "committed_tokens_per_s": _sum_over_ranks(n_pos * n_blocks, dist) / _max_over_ranks(e2e_s, dist)}
    else:
        h_tokens = torch.empty(n_pos, dtype=torch.int32).pin_memory()
        h_masked = torch.empty(n_pos, dtype=torch.uint8).pin_memory()
        h_in = x_fixed.cpu().pin_memory()
        o_tokens = torch.empty(n_pos, dtype=torch.int32).pin_memory()
        o_masked = torch.empty(n_pos, dtype=torch.uint8).pin_memory()
        o_x = torch.empty((n_pos, D.hidden), dtype=torch.float32).pin_memory()
        h_draft = draft.cpu().pin_memory() if kind == "accept" else None
        o_len = torch.empty(1, dtype=torch.int32).pin_memory()
        h_tokens.fill_(D.mask_id)
        h_masked.fill_(1)

        def e2e_step():
            x_fixed.copy_(h_in, non_blocking=True)
            if kind == "accept":
                draft.copy_(h_draft, non_blocking=True)
            elif not sp.one_layer:
                tokens.copy_(h_tokens, non_blocking=True)
                masked.copy_(h_masked, non_blocking=True)
            step(0)
            if sp.one_layer:
                o_x.copy_(x_out, non_blocking=True)
            elif kind == "accept":
                o_tokens.copy_(acc_out["tokens"], non_blocking=True)
                o_len.copy_(acc_out["accept_len"][:1], non_blocking=True)
            else:
                o_tokens.copy_(tokens, non_blocking=True)
                o_masked.copy_(masked, non_blocking=True)
            torch.cuda.synchronize()

        e2e_step()                               # untimed: first use of the buffers
        _barrier(dist)
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        e2e_s = time.perf_counter() - t0
        e2e_units = n_pos * K
        if sp.one_layer:
            h2d, d2h = n_pos * D.hidden * 4, n_pos * D.hidden * 4
        elif kind == "accept":
            h2d, d2h = n_pos * D.hidden * 4 + n_pos * 4, n_pos * 4 + 4
        else:
            h2d = n_pos * 4 + n_pos + n_pos * D.hidden * 4
            d2h = n_pos * 4 + n_pos
        e2e_extra = {"entry_point": {"layer": "clover_moe_block_step", "zipf_layer": "clover_moe_block_step",
                                     "int4_layer": "clover_moe_block_step", "head": "clover_lmhead_unmask",
                                     "accept": "clover_lmhead_accept"}[kind]}

    # collectives: every rank takes part before rank 0 alone reports
    value = replica_throughput(n_pos * K, ms * 1e-3, dist)
    e2e_value = replica_throughput(e2e_units, e2e_s, dist)
    committed_s = replica_throughput(committed, ms * 1e-3, dist) if sp.full else None
    ms_max = _max_over_ranks(ms, dist)
    if rank != 0:
        return
    csum = clk.summary()
    fused = n_pos <= 32
    per_layer = 1 if fused else 3         # fused layer kernel, or route + experts + combine
    if sp.full:
        # embed, layers, the last deferred combine, norm + a head launch and its merge launch
        # per 256 positions
        launches_per_step = 1 + per_layer * n_layers + (1 if fused else 0) + 1 + 2 * ((n_pos + 255) // 256)
    elif sp.one_layer:
        launches_per_step = per_layer
    else:
        launches_per_step = 3          # norm, head, merge
    roof_kernel = ("k_rmsnorm + k_head + k_head_merge (head statistics and unmask)" if kind == "head"
                   else "k_rmsnorm + k_head<accept> + k_head_merge<accept> (head statistics, entropy and the "
                        "accept test)"
                   if kind == "accept"
                   else "k_layer (routing + grouped SwiGLU experts + combine, one launch per MoE layer)"
                   if fused else "k_expert (grouped SwiGLU experts + combine, one launch per MoE layer)")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded random-init bf16 weights of the Clover shapes)",
        "config": base_config(kind, ws_n),
        "step_measurement": {
            "timed_steps": ("K steps from K copies of the block at evenly spaced points of its denoising loop "
                            f"(committed slots at entry: {phases})") if sp.full else "K identical calls",
            "mean_unique_experts_per_layer": u_mean,
            "algorithmic_bytes_per_step": step_bytes,
            "step_hbm_gbs": step_bytes / (ms_max / K * 1e-3) / 1e9,
            "step_roofline_frac": step_bytes / (ms_max / K * 1e-3) / 1e9 / peak,
            "committed_tokens_per_s": committed_s},
        "roofline": {"kernel": roof_kernel, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": _expert_traffic(u_mean, fused, sp.q4) if not sp.head_like else None,
                     "launches": len(durs),
                     "mean_launch_us": float(np.mean(durs)) * 1e3, "share_of_step": share,
                     "timing": "CUDA events around every launch of the kernel in a second pass over the same K "
                               "steps; events between launches stop each launch from overlapping its "
                               "predecessor, so the per-launch time is an upper bound (that pass: "
                               f"{ms_instr / K:.3f} ms per step against {ms_max / K:.3f} without events)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                **e2e_extra},
        "gpu_launches": K * launches_per_step,
        "clocks": csum,
    }
    if not args.no_cpu_baseline and ws_n == 1 and kind in ("step", "layer", "head"):
        line["cpu_baseline"] = cpu_baseline(sp, layers)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-1core", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--workload", default="step", choices=sorted(WORKLOADS),
                    help="step (default, the headline): full 40-layer block step; layer / head / zipf: the other "
                         "configurations")
    args = ap.parse_args()
    if args.oracle_1core:
        _oracle_1core_child(args.workload)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
