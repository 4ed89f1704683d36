#!/usr/bin/env python3
"""Throughput of the P-EAGLE parallel draft step on GB300.

One step = one pass of the decode hot path over one synthetic batch: the
parallel draft step (fc/fc_norm, masked-depth inputs, rotary-by-position,
depth-masked attention over context + chain, MLP, draft-vocab head and
argmax) followed by greedy verify/accept, all through the C ABI.

Workload (default): bf16 batched decode, 64 requests with context lengths
uniform in [512, 8192], K = 8 depths, target hidden 4096 with 3 aux layers,
one Llama-3-8B-sized draft layer (32 q / 8 kv heads x 128, SwiGLU 14336),
draft vocab 32000. Weights and inputs are seeded synthetic data; every step
streams 849 MB of weights and about 1.2 GB of context K/V, far more than the
129 MB L2, so no L2 flush is needed between steps.

Metric: drafted tokens/s = B * K / step time (whole job over all ranks).
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload NAME]
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "drafted tokens/s per P-EAGLE draft step"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "decode_b64_ragged_k8"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
OP_IDS = {"fc": 0, "qkv": 1, "attn": 2, "o_proj": 3, "gate_up": 4, "down": 5, "lm_head": 6}
# timed steps when --steps is not given: a timed region of seconds, not
# minutes (the 32768-token training step takes about 0.2 s)
DEFAULT_STEPS = {"train_n4096_k4": 1000, "train_n32768_k8": 100}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 3000 for decode, fewer for the training workloads)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="bound on the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--backward", action="store_true",
                    help="training workloads: time the forward + backward (gradients of every weight)")
    ap.add_argument("--probe-steps", type=int, default=None,
                    help="steps of each per-op timing pass (default: --steps, at least 300, at most 2000)")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the end-to-end pass (default: as --probe-steps)")
    ap.add_argument("--no-aux-ops", action="store_true",
                    help="decode workloads: skip the closed-loop / verification / COD latency pass")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(args.workload, 3000)
    return args


def pass_steps(args):
    """(per-op probe steps, end-to-end steps): long enough for several clock
    samples under load unless given explicitly (short runs under a profiler)."""
    probe = args.probe_steps if args.probe_steps else min(max(args.steps, 300), 2000)
    e2e = args.e2e_steps if args.e2e_steps else probe
    return max(1, probe), max(1, e2e)


# ----------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's value (the job is as slow as its slowest
    rank); identity without a process group."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, B, K, ms_step):
    """Drafted tokens/s of the whole job: every rank drafts B*K per step."""
    return world * B * K / (ms_step / 1000.0)


def algorithmic_bytes(wl, B, kv_lens):
    """Bytes each operation must move at minimum in one step, summed over the
    layers: weights once, activations in, fp32 results out; attention reads
    the context K/V once. Layer 0's QKV reads only the B anchor rows (the
    masked rows share one precomputed q/k/v); later layers read all rows."""
    es = 2 if wl.dtype == "bf16" else 4
    K, H, I, V, L = wl.K, wl.hidden, wl.intermediate, wl.vocab, wl.num_layers
    AHt = wl.num_aux * wl.target_hidden
    QKV, nqhd = wl.qkv_out, wl.num_q_heads * wl.head_dim
    rows = B * K
    kv = int(np.sum(kv_lens)) * wl.num_kv_heads * wl.head_dim * 2 * es
    return {
        "fc": es * (H * AHt + B * AHt) + 4 * B * H,
        "qkv": (es * (QKV * 2 * H + B * 2 * H) + 4 * B * QKV
                + (L - 1) * (es * (QKV * H + rows * H) + 4 * rows * QKV)),
        "attn": L * (kv + 2 * rows * nqhd * es + rows * 2 * wl.num_kv_heads * wl.head_dim * es),
        "o_proj": L * (es * (H * nqhd + rows * nqhd) + 4 * rows * H),
        "gate_up": L * (es * (2 * I * H + rows * H) + 2 * rows * I),
        "down": L * (es * (H * I + rows * I) + 4 * rows * H),
        "lm_head": es * (V * H + rows * H) + 4 * rows * V,
    }


def algorithmic_flops(wl, B):
    """Multiply-add flops of each contraction in one step (2 per MAC), over
    the rows that exist: B anchor rows for fc and layer-0 QKV, B*K rows for
    the rest."""
    K, H, I, V, L = wl.K, wl.hidden, wl.intermediate, wl.vocab, wl.num_layers
    AHt = wl.num_aux * wl.target_hidden
    QKV, nqhd = wl.qkv_out, wl.num_q_heads * wl.head_dim
    rows = B * K
    return {
        "fc": 2.0 * B * H * AHt,
        "qkv": 2.0 * B * QKV * 2 * H + (L - 1) * 2.0 * rows * QKV * H,
        "o_proj": 2.0 * L * rows * H * nqhd,
        "gate_up": 2.0 * L * rows * 2 * I * H,
        "down": 2.0 * L * rows * H * I,
        "lm_head": 2.0 * rows * V * H,
    }


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


def _code_only(text):
    """C++/CUDA source without comments and blank space: edits to comments
    leave the kernels, and so the digest, unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":   # string / char literal, copied as is
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(root=None):
    """Digest of what the recorded ncu counters depend on: the kernel sources
    and the public header they include (code only), plus the nvcc target
    and flags the library is built with."""
    root = root or ROOT
    h = hashlib.sha256()
    pkg = os.path.join(root, "eagle_speculative_drafting_gb300")
    csrc = os.path.join(pkg, "csrc")
    files = [(f, os.path.join(csrc, f)) for f in sorted(os.listdir(csrc))]
    files.append(("include/peagle.h", os.path.join(root, "include", "peagle.h")))
    for name, path in files:
        with open(path, encoding="utf-8") as fh:
            h.update(name.encode() + b"\0" + _code_only(fh.read()).encode())
    build = os.path.join(pkg, "_build.py")
    if os.path.exists(build):
        with open(build, encoding="utf-8") as fh:
            text = fh.read()
        for key in ("ARCH", "FLAGS"):
            for ln in text.splitlines():
                if ln.startswith(key + " ="):
                    h.update(ln.encode())
    return h.hexdigest()[:16]


def graph_replay(step, d, targets, steps, dist):
    """Times `steps` replays of one draft step + verify captured as a CUDA
    graph; None without a GPU, or {"error": ...} if the capture failed."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step(d, targets, torch.cuda.current_stream())   # warm the side stream once
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step(d, targets, torch.cuda.current_stream())
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            g.replay()
        e1.record(s)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda") / steps
        return {"ms_per_step": ms, "replays": steps}
    except Exception as exc:   # reported in the JSON line, never fatal
        torch.cuda.synchronize()
        return {"error": str(exc).splitlines()[0][:200]}


def recorded_traffic(op, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{workload}:{op}")
    if not e or e.get("source_digest") != source_digest():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle leg
def oracle_leg(wl, W, inp, seconds, warm=1, max_steps=None):
    """Times whole oracle draft steps (all requests, all depths) on the host
    until `seconds` have passed; returns (tokens/s, steps, elapsed, cores)."""
    from oracle import peagle_oracle as O
    model = O.DraftModel(O.model_config(wl), W)
    args = (inp["aux"], inp["anchor_tokens"], inp["anchor_pos"], inp["k_cache"], inp["v_cache"],
            inp["kv_offsets"], inp["kv_lens"], wl.K)
    for _ in range(warm):
        O.draft_step(model, *args)
    steps, t0 = 0, time.perf_counter()
    while True:
        O.draft_step(model, *args)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_steps and steps >= max_steps):
            break
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    return wl.batch * wl.K * steps / el, steps, el, cores


def oracle_train_leg(wl, W, inp, seconds, max_steps=None, backward=False):
    """The oracle on the host cores over a bounded sample of a training
    workload: the forward of its shortest conversation (exact on its own:
    conversations never attend to one another), or, for the backward, the
    float64 autograd gradients of every weight over the first <= 128 tokens
    of that conversation as a packed sequence of their own. Returns
    (rows/s, steps, seconds, cores, sample)."""
    from oracle import peagle_oracle as O
    model = O.DraftModel(O.model_config(wl), W)
    cu = inp["cu_seqlens"]
    conv = int(np.argmin(np.diff(cu)))
    K, r, rmin, seed = inp["K"], inp["r"], inp["r_min"], inp["seed"]
    if not backward:
        fwd = {k: inp[k] for k in ("aux", "input_ids", "position_ids", "cu_seqlens", "labels", "loss_mask")}
        kw = dict(K=K, r=r, r_min=rmin, seed=seed, conversations=[conv], keep_logits=False)
        res = O.parallel_forward(model, **fwd, **kw)
        rows = int(np.sum(res["row_argmax"] >= 0))
        run = lambda: O.parallel_forward(model, **fwd, **kw)
        what = f"oracle forwards of conversation {conv} ({int(cu[conv + 1] - cu[conv])} tokens, {rows} rows)"
    else:
        a = int(cu[conv])
        b = min(int(cu[conv + 1]), a + 128)
        sub = dict(aux=inp["aux"][a:b], input_ids=np.asarray(inp["input_ids"])[a:b],
                   position_ids=np.asarray(inp["position_ids"])[a:b], cu_seqlens=np.array([0, b - a]),
                   labels=np.asarray(inp["labels"])[a:b], loss_mask=None)
        rows = int(sum(O.cod_counts(b - a, K, r, rmin)))
        run = lambda: O.parallel_grads(model, **sub, K=K, r=r, r_min=rmin, seed=seed,
                                       depth_decay=inp["depth_decay"])
        what = (f"oracle backward passes (float64 autograd gradients of every weight) over the first {b - a} "
                f"tokens of conversation {conv} as a packed sequence of their own ({rows} rows)")
    steps, t0 = 0, time.perf_counter()
    while True:
        run()
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_steps and steps >= max_steps):
            break
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    return rows * steps / el, steps, el, cores, f"{steps} {what} in {el:.1f} s"


def run_reference_train(args, wl):
    """Oracle timing of the training-shaped forward on whole sampled
    conversations (exact on their own: conversations never attend to one
    another), reported as rows of those conversations per second."""
    import synth
    W = synth.make_weights(wl)
    inp = synth.make_train_inputs(wl)
    v, steps, el, cores, sample = oracle_train_leg(wl, W, inp, min(60.0, args.cpu_seconds * 2),
                                                   max_steps=args.steps, backward=args.backward)
    metric = "training rows/s per P-EAGLE forward + backward" if args.backward else TRAIN_METRIC
    line = {"impl": "reference", "metric": metric, "value": v, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": 1, "ms_per_step": 1000.0 * el / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name},
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if wl.kind == "train":
        return run_reference_train(args, wl)
    import synth
    W = synth.make_weights(wl)
    inp = synth.make_decode_inputs(wl)
    # every step is one whole oracle draft step; the number of steps is bounded
    # so the run stays within a few minutes whatever --steps asks for
    budget = min(180.0, 3.0 + 0.5 * args.steps)
    v, steps, el, cores = oracle_leg(wl, W, inp, seconds=min(budget, 60.0), warm=min(args.warmup, 1),
                                     max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": min(args.warmup, 1), "ms_per_step": 1000.0 * el / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{steps} whole float64 oracle draft steps ({wl.batch} request x "
                                   f"{wl.K} depths each) in {el:.1f} s"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl):
    return {"workload": wl.name, "batch": wl.batch, "K": wl.K,
            "kv_context": wl.kv_len or list(wl.kv_len_range), "hidden": wl.hidden,
            "target_hidden": wl.target_hidden, "num_aux": wl.num_aux, "layers": wl.num_layers,
            "heads": f"{wl.num_q_heads}q/{wl.num_kv_heads}kv x {wl.head_dim}",
            "intermediate": wl.intermediate, "draft_vocab": wl.vocab,
            "l2": "weights larger than L2 (streamed every step), no flush",
            "parallelism": "replicas (independent requests per GPU)"}


# ---------------------------------------- the rows around the draft step
LOOP_ROUNDS = 64


def aux_ops(pe, synth, marshal, wl, model, d, inp, stream, rounds=LOOP_ROUNDS):
    """Latency of the rows around the draft step, each timed with CUDA events
    on its stream after the headline passes: the closed draft -> verify ->
    next-context loop over the workload's requests (a synthetic target stands
    in: aux states of the new rows, and targets agreeing with the drafts for
    a truncated-geometric number of depths; it runs outside the timed
    events), greedy and stochastic verification, and COD selection at the
    two training shapes."""
    import torch
    from eagle_speculative_drafting_gb300.loop import DraftLoop
    B, K, V = wl.batch, wl.K, wl.vocab
    Vd = model.cfg.draft_vocab
    dev = "cuda"
    ev = lambda: torch.cuda.Event(enable_timing=True)
    out = {}
    # ---- closed loop
    loop = DraftLoop(model, K, d["k_cache"], d["v_cache"], d["kv_offsets"], d["kv_lens"], int(inp["kv_capacity"]),
                     stream)
    loop.start(inp["anchor_tokens"], inp["anchor_pos"])
    g = torch.Generator(device=dev).manual_seed(7)
    aux_rows = torch.randn(B * (K + 1), wl.num_aux * wl.target_hidden, device=dev, generator=g).to(marshal.tdtype(wl))
    ar = torch.arange(K + 1, device=dev)
    zero_col = torch.zeros(B, 1, dtype=torch.int32, device=dev)
    t_draft = t_rest = 0.0
    kept = 0
    torch.cuda.synchronize()
    for r in range(rounds):
        e0, e1, e2, e3 = ev(), ev(), ev(), ev()
        e0.record(stream)
        drafts = loop.draft(aux_rows[:loop.total_new])
        e1.record(stream)
        a = torch.from_numpy(synth.draw_accept_lengths(wl, B, K, salt=r + 1)).to(dev)
        ext = torch.cat([drafts, zero_col], 1)
        tgt = torch.where(ar[None] < a[:, None], ext, (ext + 1) % V).to(torch.int32).contiguous()
        torch.cuda.synchronize()
        e2.record(stream)
        acc, _ = loop.verify_greedy(tgt)   # verify, next rows, and the host read that sizes the next round
        e3.record(stream)
        torch.cuda.synchronize()
        t_draft += e0.elapsed_time(e1)
        t_rest += e2.elapsed_time(e3)
        kept += int(acc.sum().item()) + B
    ms = (t_draft + t_rest) / rounds
    out["closed_loop"] = {
        "rounds": rounds, "requests": B, "K": K, "ms_per_round": ms, "draft_ms": t_draft / rounds,
        "verify_next_context_ms": t_rest / rounds, "mean_accept": kept / (rounds * B) - 1.0,
        "drafted_tokens_per_s": B * K / (ms / 1000.0), "kept_tokens_per_s": kept / ((t_draft + t_rest) / 1000.0),
        "device_status": pe.peagle_get_device_status(model.handle)}

    def per_call_us(fn, n):
        fn()
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return 1000.0 * e0.elapsed_time(e1) / n

    # ---- greedy and stochastic verification of B x K drafts
    dr = torch.randint(0, Vd, (B, K), dtype=torch.int32, device=dev, generator=g)
    tg = torch.randint(0, Vd, (B, K + 1), dtype=torch.int32, device=dev, generator=g)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    out["verify_accept_us"] = per_call_us(lambda: pe.peagle_verify_accept(B, K, dr, tg, acc, nxt, stream), 1000)
    logits = torch.randn(B, K + 1, Vd, device=dev, generator=g) * 3.0
    p = torch.softmax(logits + 0.5 * torch.randn(B, K + 1, Vd, device=dev, generator=g), -1).contiguous()
    q = torch.softmax(logits[:, :K], -1).contiguous()
    dq = torch.multinomial(q.view(-1, Vd), 1, generator=g).view(B, K).to(torch.int32).contiguous()
    u = torch.rand(B, K, device=dev, generator=g)
    draws = torch.randint(0, 2 ** 31 - 1, (B,), dtype=torch.int32, device=dev, generator=g)
    out["verify_sample_us"] = per_call_us(
        lambda: pe.peagle_verify_sample(B, K, Vd, dq, q, p, u, draws, acc, nxt, stream), 200)
    out["verify_sample_shape"] = f"B={B} K={K} V={Vd}"
    # ---- COD selection at the training shapes (r = 0.7, r_min = 0.2)
    cod = {}
    for n, Kc in ((4096, 4), (32768, 8)):
        R = sum(pe.peagle_cod_counts(n, Kc, 0.7, 0.2))
        idx = torch.empty(R, dtype=torch.int32, device=dev)
        row_of = torch.empty(Kc * n, dtype=torch.int32, device=dev)
        wsb = pe.peagle_cod_select_workspace_size(n, Kc)
        wsc = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        cod[f"n{n}_k{Kc}"] = per_call_us(
            lambda: pe.peagle_cod_select(n, Kc, 0.7, 0.2, 0x5EED, idx, row_of, wsc, wsb, stream), 50)
    out["cod_select_us"] = cod
    out["timing"] = "CUDA events on the launching stream, after the headline passes"
    # ---- checkpoint I/O: the model's device weights saved in vLLM's layout
    # (safetensors + config.json) to a temporary directory and loaded into
    # fresh device buffers (host wall clock; the files sit in the page cache)
    import shutil
    import tempfile
    from eagle_speculative_drafting_gb300.model import load_checkpoint
    tmp = tempfile.mkdtemp(prefix="peagle_ckpt_")
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        model.save_checkpoint(tmp)
        t1 = time.perf_counter()
        m2 = load_checkpoint(tmp)
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        m2.close()
        nbytes = sum(os.path.getsize(os.path.join(tmp, f)) for f in os.listdir(tmp))
        out["checkpoint"] = {"bytes": nbytes, "save_s": t1 - t0, "load_s": t2 - t1,
                             "save_gbs": nbytes / (t1 - t0) / 1e9, "load_gbs": nbytes / (t2 - t1) / 1e9,
                             "timing": "host wall clock, device memory <-> files in a temporary directory"}
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return out


# ------------------------------------------------------ training-shaped pass
TRAIN_METRIC = "drafted depth-rows/s per P-EAGLE parallel forward"
TRAIN_OPS = {"fc": 0, "qkv": 1, "attn": 2, "o_proj": 3, "gate_up": 4, "down": 5, "lm_head": 6, "ce": 9}
BWD_GEMM_OP = 10   # every contraction of the parallel backward


def train_flops(wl, n, R, pairs):
    """Algorithmic flops per forward of each operation (dense products only
    over the rows that exist; attention over allowed key pairs)."""
    H, I, V = wl.hidden, wl.intermediate, wl.vocab
    AHt, QKV, nqhd, L = wl.num_aux * wl.target_hidden, wl.qkv_out, wl.num_q_heads * wl.head_dim, wl.num_layers
    return {
        "fc": 2.0 * n * H * AHt,
        "qkv": 2.0 * n * QKV * 2 * H + 2.0 * (L - 1) * R * QKV * H,
        "attn": 4.0 * wl.head_dim * wl.num_q_heads * pairs * L,
        "o_proj": 2.0 * L * R * H * nqhd,
        "gate_up": 2.0 * L * R * 2 * I * H,
        "down": 2.0 * L * R * H * I,
        "lm_head": 2.0 * R * V * H,
        "ce": 0.0,
    }


def allowed_pairs(indices, counts, cu):
    """Key pairs the depth-masked attention scores: row (i, d) reads the
    depth-0 rows start(i)..i and its d chain rows."""
    cu = np.asarray(cu, dtype=np.int64)
    n = int(cu[-1])
    start = np.zeros(n, dtype=np.int64)
    for c in range(len(cu) - 1):
        start[cu[c]:cu[c + 1]] = cu[c]
    depth = np.repeat(np.arange(len(counts)), counts)
    idx = np.asarray(indices, dtype=np.int64)
    return int(np.sum(idx - start[idx] + 1 + depth))


def run_train(args, wl):
    """Training-shaped forward. With N ranks every rank runs its own packed
    sequence of the workload's shape (data parallel, weak scaling); the ranks
    exchange their per-depth sums in one NCCL all-reduce per step and every
    rank combines them into the batch loss."""
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    import eagle_speculative_drafting_gb300 as pe
    import synth
    from eagle_speculative_drafting_gb300 import dp, marshal

    W = synth.make_weights(wl)
    # sequence `rank` of the global batch: its own conversations and tokens
    inp = synth.make_train_inputs(wl.scaled(seed=wl.seed + 7919 * rank) if rank else wl)
    model = marshal.make_model(wl, W)
    d = marshal.upload_train(wl, inp)
    n, K, r, rmin = wl.n_tokens, inp["K"], inp["r"], inp["r_min"]
    seed = dp.sequence_seed(inp["seed"], rank) if world > 1 else inp["seed"]
    counts = pe.peagle_cod_counts(n, K, r, rmin)
    R = sum(counts)
    idx = torch.empty(R, dtype=torch.int32, device="cuda")
    pe.peagle_cod_select(n, K, r, rmin, seed, idx)
    pairs = allowed_pairs(idx.cpu().numpy(), counts, inp["cu_seqlens"])
    flops = train_flops(wl, n, R, pairs)
    dev = dict(device="cuda")
    outs = [torch.empty(K, dtype=torch.float32, **dev), torch.empty(K, dtype=torch.float32, **dev),
            torch.empty(K, dtype=torch.int32, **dev), torch.empty(1, dtype=torch.float32, **dev)]
    nbytes = pe.peagle_parallel_forward_workspace_size(model.handle, n, K, r, rmin)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    S = len(inp["cu_seqlens"]) - 1
    sums = torch.zeros(3 * K, dtype=torch.float64, **dev)

    def step(dd):
        if dist is None:
            pe.peagle_parallel_forward(model.handle, n, dd["aux"], dd["input_ids"], dd["position_ids"],
                                       dd["cu_seqlens"], S, dd["labels"], None, K, r, rmin, seed,
                                       inp["depth_decay"], *outs, None, None, None, ws, nbytes, stream)
            return
        # data parallel: this rank's sequence adds its depth sums, one
        # all-reduce, then the batch loss on every rank
        sums.zero_()
        pe.peagle_parallel_forward(model.handle, n, dd["aux"], dd["input_ids"], dd["position_ids"],
                                   dd["cu_seqlens"], S, dd["labels"], None, K, r, rmin, seed,
                                   inp["depth_decay"], *outs, None, None, None, ws, nbytes, stream,
                                   depth_sums=sums)
        dp.allreduce_depth_sums(sums, dist)
        pe.peagle_combine_depth_sums(K, inp["depth_decay"], sums, *outs, stream)

    for _ in range(max(args.warmup, 3)):
        step(d)
    torch.cuda.synchronize()
    clk = ClockSampler(local).__enter__()   # through the probe, timed and e2e passes
    shares = {}
    for name, op in TRAIN_OPS.items():
        pe.peagle_probe_begin(op, 4096)
        for _ in range(2):
            step(d)
        ms = pe.peagle_probe_end(4096)
        shares[name] = float(np.sum(ms)) / 2.0 if ms else 0.0
    dom = max(shares, key=shares.get)
    launches0 = pe.peagle_kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step(d)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    launches = pe.peagle_kernel_launches() - launches0
    ms_step = max_over_ranks(e0.elapsed_time(e1), dist, "cuda") / args.steps
    # the dominant op, timed with CUDA events around its launches in a pass
    # of its own (events between PDL-chained kernels serialize them)
    probe_steps = max(1, min(args.steps, 10))
    pe.peagle_probe_begin(TRAIN_OPS[dom], 1 << 18)
    for _ in range(probe_steps):
        step(d)
    torch.cuda.synchronize()
    dom_ms = pe.peagle_probe_end(1 << 18)
    # end to end: the step's inputs from pinned host memory, the loss back
    keys = ("aux", "input_ids", "position_ids", "cu_seqlens", "labels")
    h_in = {k: d[k].cpu().pin_memory() for k in keys}
    h_out = torch.empty(3 * K + 1, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)
    e_steps = max(1, min(args.steps, 50))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(e_steps):
        for k in keys:
            d[k].copy_(h_in[k], non_blocking=True)
        step(d)
        h_out[:K].copy_(outs[0], non_blocking=True)
        h_out[K:2 * K].copy_(outs[1], non_blocking=True)
        h_out[2 * K:3 * K].copy_(outs[2].float(), non_blocking=True)
        h_out[3 * K:].copy_(outs[3], non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    e2e_ms = max_over_ranks(e2.elapsed_time(e3) / e_steps, dist, "cuda")
    status = pe.peagle_get_device_status(model.handle)
    if rank != 0:
        model.close()
        if dist:
            dist.destroy_process_group()
        return
    _, _, peak, src = measured_peaks()
    src += " (sustained)"
    total_dom_ms = float(np.sum(dom_ms)) / probe_steps if dom_ms else None
    achieved = flops[dom] / (total_dom_ms / 1000.0) / 1e12 if total_dom_ms else None
    line = {
        "metric": TRAIN_METRIC, "value": world * R / (ms_step / 1000.0), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic",
        "config": {"workload": wl.name, "n_tokens": n, "conversations": S, "K": K, "rows": R,
                   "cod_counts": counts, "layers": wl.num_layers, "hidden": wl.hidden,
                   "heads": f"{wl.num_q_heads}q/{wl.num_kv_heads}kv x {wl.head_dim}",
                   "intermediate": wl.intermediate, "draft_vocab": wl.vocab,
                   "l2": "activations and weights far larger than L2, no flush",
                   "parallelism": f"data parallel over {world} rank(s): one packed sequence each, "
                                  "one all-reduce of the per-depth sums per step"},
        "gpu_launches": int(launches),
        "e2e": {"value": world * R / (e2e_ms / 1000.0), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_source": src, "unit": "TFLOP/s",
                     "frac": achieved / peak if achieved else None, "traffic": None,
                     "algorithmic_flops_per_step": flops[dom], "ms_per_step": total_dom_ms},
        "step_shares_ms": {k: round(v, 4) for k, v in shares.items()},
        "flops_per_step": {k: v for k, v in flops.items()},
        "device_status": status,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        v, _, _, cores, sample = oracle_train_leg(wl, W, inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    model.close()
    if dist:
        dist.destroy_process_group()


def run_backward(args, wl):
    """Forward + backward of the training-shaped pass on one GPU: the loss
    and the gradients of every weight but the embedding, per packed
    sequence. Metric: training rows (all depths) per second."""
    import torch
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_drafting_gb300 as pe
    import synth
    from eagle_speculative_drafting_gb300 import marshal
    from eagle_speculative_drafting_gb300.model import weight_shapes, weights_struct

    W = synth.make_weights(wl)
    inp = synth.make_train_inputs(wl)
    model = marshal.make_model(wl, W)
    d = marshal.upload_train(wl, inp)
    n, K, r, rmin, seed = wl.n_tokens, inp["K"], inp["r"], inp["r_min"], inp["seed"]
    R = sum(pe.peagle_cod_counts(n, K, r, rmin))
    nbytes = pe.peagle_parallel_backward_workspace_size(model.handle, n, K, r, rmin)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    shapes = weight_shapes(model.cfg)
    f32 = dict(dtype=torch.float32, device="cuda")
    grads = {k: torch.empty(shapes[k], **f32) for k in ("fc_w", "fc_norm_w", "mask_hidden", "final_norm_w",
                                                           "lm_head_w")}
    grads["layers"] = [{k: (None if sh is None else torch.empty(sh, **f32)) for k, sh in L.items()}
                       for L in shapes["layers"]]
    gw, keep = weights_struct(grads)
    loss = torch.empty(1, **f32)
    S = len(inp["cu_seqlens"]) - 1
    stream = torch.cuda.current_stream()

    def step():
        pe.peagle_parallel_backward(model.handle, n, d["aux"], d["input_ids"], d["position_ids"], d["cu_seqlens"],
                                    S, d["labels"], None, K, r, rmin, seed, inp["depth_decay"], loss, gw, ws,
                                    nbytes, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(local).__enter__()
    launches0 = pe.peagle_kernel_launches()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = pe.peagle_kernel_launches() - launches0
    ms = e0.elapsed_time(e1) / args.steps
    # the pass's contractions (the forward again, then dX and dW of each),
    # timed with CUDA events around each launch in a pass of their own
    probe_steps = max(1, min(args.steps, 5))
    pe.peagle_probe_begin(BWD_GEMM_OP, 1 << 16)
    for _ in range(probe_steps):
        step()
    torch.cuda.synchronize()
    gemm_ms = float(np.sum(pe.peagle_probe_end(1 << 16))) / probe_steps
    f = train_flops(wl, n, R, 0)
    dense = sum(f[k] for k in ("fc", "qkv", "o_proj", "gate_up", "down", "lm_head"))
    gemm_flops = 3.0 * dense - f["fc"]   # forward, dX and dW of each; fc has no dX (aux is an input)
    _, _, peak, src = measured_peaks()
    achieved = gemm_flops / (gemm_ms / 1000.0) / 1e12 if gemm_ms > 0 else None
    # end to end: the step's inputs from pinned host memory, the loss back
    keys = ("aux", "input_ids", "position_ids", "cu_seqlens", "labels")
    h_in = {k: d[k].cpu().pin_memory() for k in keys}
    h_loss = torch.empty(1, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    e_steps = max(1, min(args.steps, 20))
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(e_steps):
        for k in keys:
            d[k].copy_(h_in[k], non_blocking=True)
        step()
        h_loss.copy_(loss, non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize()
    clk.__exit__(None, None, None)
    e2e_ms = e2.elapsed_time(e3) / e_steps
    line = {"metric": "training rows/s per P-EAGLE forward + backward", "value": R / (ms / 1000.0),
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic", "config": {"workload": wl.name, "n_tokens": n, "K": K, "rows": R,
                                            "pass": "forward + backward, gradients of every weight"},
            "gpu_launches": int(launches), "loss": float(loss.item()),
            "e2e": {"value": R / (e2e_ms / 1000.0), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": 4},
            "roofline": {"bound": "tensor", "kernel": "gemm_tc_kernel (every contraction of the pass)",
                         "achieved": achieved, "peak": peak, "peak_source": src + " (sustained)",
                         "unit": "TFLOP/s", "frac": achieved / peak if achieved else None, "traffic": None,
                         "algorithmic_flops_per_step": gemm_flops, "ms_per_step": gemm_ms,
                         "timing": f"CUDA events around each launch on its stream, {probe_steps} steps"},
            "workspace_bytes": int(nbytes), "device_status": pe.peagle_get_device_status(model.handle),
            "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        v, _, _, cores, sample = oracle_train_leg(wl, W, inp, args.cpu_seconds, backward=True)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    model.close()


# ------------------------------------------------------------------- ours
def main():
    args = parse_args()
    import synth
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    if wl.kind == "train":
        return run_backward(args, wl) if args.backward else run_train(args, wl)

    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    import eagle_speculative_drafting_gb300 as pe
    from eagle_speculative_drafting_gb300 import marshal

    W = synth.make_weights(wl)
    # spare cache rows per request for the closed loop's appended rows
    inp = synth.make_decode_inputs(wl, spare=wl.K + LOOP_ROUNDS * (wl.K + 1))
    model = marshal.make_model(wl, W)
    d = marshal.upload_decode(wl, inp)
    B, K = wl.batch, wl.K
    kv_cap = int(inp["kv_capacity"])
    max_kv = int(np.max(inp["kv_lens"]))
    drafts = torch.empty((B, K), dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    ws_bytes = pe.peagle_draft_step_workspace_size(model.handle, B, K, max_kv)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(dd, targets, on=None):
        st = stream if on is None else on
        pe.peagle_draft_step(model.handle, B, K, dd["aux"], dd["anchor_tokens"], dd["anchor_pos"],
                             dd["k_cache"], dd["v_cache"], dd["kv_offsets"], dd["kv_lens"], kv_cap,
                             max_kv, 0, drafts, None, ws, ws_bytes, st)
        pe.peagle_verify_accept(B, K, drafts, targets, acc, nxt, st)

    # targets whose agreement with the drafts has geometric(0.7) length
    step(d, torch.zeros((B, K + 1), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    accept = synth.draw_accept_lengths(wl, B, K)
    tgt_np = synth.make_targets_with_accept(wl, drafts.cpu().numpy(), accept)
    targets = torch.from_numpy(tgt_np).cuda()

    for _ in range(max(args.warmup, 3)):
        step(d, targets)
    torch.cuda.synchronize()

    abytes = algorithmic_bytes(wl, B, inp["kv_lens"])
    aflops = algorithmic_flops(wl, B)
    hbm_peak, tc_peak, _, peak_src = measured_peaks()
    # Clocks are sampled from here to the end of the end-to-end pass: the
    # per-op probe pass, the timed region, the dominant-kernel pass and the
    # end-to-end pass all run the same steps under load.
    clk = ClockSampler(local).__enter__()

    # ---- per-op time: CUDA events around every launch of one op class
    # (the contraction's kernel, or the attention's split kernel) on its own
    # launch stream, one class at a time
    probe_steps, e_steps = pass_steps(args)
    per_op_ms = {}
    for name, op in OP_IDS.items():
        cap = probe_steps * wl.num_layers + 8
        pe.peagle_probe_begin(op, cap)
        for _ in range(probe_steps):
            step(d, targets)
        torch.cuda.synchronize()
        ms = pe.peagle_probe_end(cap)
        per_op_ms[name] = (float(np.sum(ms)) / probe_steps if ms else 0.0, len(ms) / probe_steps if ms else 0)
    shares = {k: v[0] for k, v in per_op_ms.items()}
    dom = max(shares, key=shares.get)

    # ---- timed region: K steps, device events, barrier + sync both sides.
    # No probe events inside it: an event recorded between two PDL-chained
    # kernels serializes them, so the per-op times come from the pass above.
    launches0 = pe.peagle_kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step(d, targets)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    launches = pe.peagle_kernel_launches() - launches0
    ms_total = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    ms_step = ms_total / args.steps
    value = job_throughput(world, B, K, ms_step)

    # ---- the same step captured once as a CUDA graph and replayed (the
    # launches are recorded with their programmatic dependencies)
    graph = graph_replay(step, d, targets, args.steps, dist)
    if graph is not None and "ms_per_step" in graph:
        graph["value"] = job_throughput(world, B, K, graph["ms_per_step"])
        graph["unit"] = UNIT

    # ---- end to end through the public API with host buffers: each step's
    # inputs leave one pinned host buffer in one copy (16-byte aligned
    # segments: aux, anchor tokens/positions, KV offsets/lengths, targets)
    # and the drafts / accept lengths / next tokens come back in one copy.
    # Both copies are the library's staging kernels (peagle_copy_to_device /
    # _to_host), which read and write the page-locked buffers from the GPU
    # and stay in the launch chain of the step
    segs = [("aux", torch.from_numpy(inp["aux"]).to(marshal.tdtype(wl))),
            ("anchor_tokens", torch.from_numpy(inp["anchor_tokens"].astype(np.int32))),
            ("anchor_pos", torch.from_numpy(inp["anchor_pos"].astype(np.int32))),
            ("kv_offsets", torch.from_numpy(inp["kv_offsets"].astype(np.int64))),
            ("kv_lens", torch.from_numpy(inp["kv_lens"].astype(np.int32))),
            ("targets", torch.from_numpy(tgt_np))]
    offs, off = {}, 0
    for k, t in segs:
        offs[k] = off
        off = (off + t.numel() * t.element_size() + 15) // 16 * 16
    h_stage = torch.zeros(off, dtype=torch.uint8).pin_memory()
    d_stage = torch.empty(off, dtype=torch.uint8, device="cuda")
    dd = dict(d)
    for k, t in segs:
        nb = t.numel() * t.element_size()
        h_stage[offs[k]:offs[k] + nb].copy_(t.contiguous().view(torch.uint8).reshape(-1))
        dd[k] = d_stage[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    dev_tgt = dd.pop("targets")
    d_out = torch.empty(B * K + 2 * B, dtype=torch.int32, device="cuda")
    h_out = torch.empty_like(d_out, device="cpu").pin_memory()
    out_drafts, out_acc, out_next = d_out[:B * K].view(B, K), d_out[B * K:B * K + B], d_out[B * K + B:]

    def step_e2e():
        pe.peagle_draft_step(model.handle, B, K, dd["aux"], dd["anchor_tokens"], dd["anchor_pos"],
                             dd["k_cache"], dd["v_cache"], dd["kv_offsets"], dd["kv_lens"], kv_cap,
                             max_kv, 0, out_drafts, None, ws, ws_bytes, stream)
        pe.peagle_verify_accept(B, K, out_drafts, dev_tgt, out_acc, out_next, stream)

    h2d = int(h_stage.numel())
    d2h = int(h_out.numel() * h_out.element_size())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(e_steps):
        pe.peagle_copy_to_device(d_stage, h_stage, h2d, stream)
        step_e2e()
        pe.peagle_copy_to_host(h_out, d_out, d2h, stream)
    e3.record(stream)
    torch.cuda.synchronize()
    # the results did come back: the host copy of the last step's drafts,
    # accept lengths and next tokens equals the device's
    e2e_outputs_match = bool(torch.equal(h_out, d_out.cpu()))
    clk.__exit__(None, None, None)
    e2e_ms = max_over_ranks(e2.elapsed_time(e3) / e_steps, dist, "cuda")
    e2e_value = job_throughput(world, B, K, e2e_ms)
    status = pe.peagle_get_device_status(model.handle)

    if rank != 0:
        model.close()
        if dist:
            dist.destroy_process_group()
        return

    # per-op roofline: every op by algorithmic bytes against HBM; the
    # contractions also by algorithmic flops against the bf16 tensor-core
    # burst peak (each op is timed alone, launch by launch)
    ops = {}
    for name, (ms, nl) in per_op_ms.items():
        if ms <= 0:
            continue
        e = {"ms_per_step": round(ms, 5), "launches_per_step": nl,
             "hbm_gbs": abytes[name] / (ms / 1000.0) / 1e9}
        e["hbm_frac"] = e["hbm_gbs"] / hbm_peak
        if name in aflops:
            e["tflops"] = aflops[name] / (ms / 1000.0) / 1e12
            e["tc_frac"] = e["tflops"] / tc_peak
        ops[name] = e
    dom_ms = per_op_ms[dom][0]
    dom_launches = max(1, per_op_ms[dom][1])
    dom_avg_ms = dom_ms / dom_launches
    achieved = (abytes[dom] / dom_launches) / (dom_avg_ms / 1000.0) / 1e9 if dom_avg_ms > 0 else None
    traffic = recorded_traffic(dom, wl.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl),
        "gpu_launches": int(launches),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "outputs_match": e2e_outputs_match,
                "copies": "staging kernels in the launch chain (page-locked host memory)"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": (achieved / hbm_peak) if achieved else None,
                     "traffic": traffic, "algorithmic_bytes": abytes[dom] / dom_launches,
                     "avg_launch_ms": dom_avg_ms,
                     "timing": f"CUDA events around each launch on its stream, {probe_steps} steps "
                               f"in a probe pass before the timed region"},
        "ops": ops,
        "graph_replay": graph,
        "tc_peak_tflops": tc_peak,
        "device_status": status,
    }
    line["clocks"] = clk.summary()
    if not args.no_aux_ops:
        line["aux_ops"] = aux_ops(pe, synth, marshal, wl, model, d, inp, stream)
    if world == 1 and not args.no_cpu_baseline:
        v, steps, el, cores = oracle_leg(wl, W, inp, seconds=args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{steps} whole float64 oracle draft steps "
                                          f"({B} requests x {K} depths each) in {el:.1f} s"}
    print(json.dumps(line), flush=True)
    model.close()
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
