#!/usr/bin/env python
"""Benchmark of the Llama decoder-layer forward on GB300.

Default workload: the 70B-shaped 8-layer stack (32 decode sequences with
contexts uniform in [1024, 16384] + 2 prefill chunks of 2048 tokens, 4128
tokens, final norm, lm_head over vocab 128256, greedy argmax).  One step is one
call of ``llama_stack_forward``: every row of the hot path.  The metric is
tokens/s per 70B-shape decoder layer (tokens x layers / step time).  The same
line carries the single-layer 70B decode (128 sequences, context U[512, 8192])
and 70B prefill (8 x 4096) results with their roofline fractions.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torch.distributed.run: each rank runs an independent
replica of the workload (sequences are independent, nothing is exchanged);
the reported time is the maximum over ranks and the value counts all ranks.
``--impl reference`` times the CPU oracle (test infrastructure, fp32) on a
bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import gc
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

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the gate_up
# GEMM at the stack's shape (4128 x 57344 x 8192) from an ncu capture of the
# current kernel (2.415 GB read + 0.183 GB written, one launch of
# `bench.py --workload gemm_gate_up`, tensor pipe 76.8% active at 1844 MHz),
# or None when the kernel has changed since that capture.
GATE_UP_DRAM_BYTES_PER_LAUNCH = 2414840576 + 183184640


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


# --------------------------------------------------------------------------- distributed plumbing


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device=None):
    """Maximum of a per-rank value (the step time) over all ranks."""
    if world == 1:
        return x
    import torch.distributed as dist
    if device is None:
        device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms_max, world):
    """Units all ranks processed per second, timed by the slowest rank
    (replicas: every rank processes its own batch of the same size)."""
    return units_per_rank * world / (ms_max / 1e3)


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- workloads


class Workload:
    """A device-resident workload and its step function."""


def setup_stack(lb, I, seed, dev, fold=False):
    spec = I.SPECS["stack_70b"]
    bl = I.make_batch(spec, seed, dev)
    layers = [I.make_layer_weights(spec, seed, l, dev) for l in range(spec.num_layers)]
    if fold:  # norm weights folded into w_qkv / w_gate_up (done once, before timing)
        layers = [lb.folded_layer_weights(w) for w in layers]
    emb, ids, lm, fn = I.make_stack_extras(spec, bl.num_tokens, seed, dev)
    caches = [I.make_kv_cache(spec, bl.num_blocks, seed, l, dev) for l in range(spec.num_layers)]
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    T, B = bl.num_tokens, bl.num_seqs
    W = Workload()
    W.spec, W.bl, W.cfg, W.batch = spec, bl, cfg, batch
    W.layers, W.emb, W.ids, W.lm, W.fn, W.caches = layers, emb, ids, lm, fn, caches
    W.hidden = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device=dev)
    W.residual = torch.empty_like(W.hidden)
    W.tokens = torch.empty(B, dtype=torch.int32, device=dev)
    W.ws = lb.alloc_workspace(lb.workspace_size(cfg, T, B, batch.max_seq_len, spec.vocab), dev)
    kcs = [c[0] for c in caches]
    vcs = [c[1] for c in caches]

    def step(stream=None, batch=None, ids=None, tokens=None):
        lb.stack_forward(cfg, layers, fn, lm, batch or W.batch, W.hidden, W.residual, kcs, vcs,
                         W.tokens if tokens is None else tokens, W.ws, embed=emb,
                         input_ids=W.ids if ids is None else ids, stream=stream)

    W.step = step
    W.tokens_per_step = T
    W.layers_n = spec.num_layers
    return W


def setup_layer(lb, I, name, seed, dev, weights=None, fold=False):
    spec = I.SPECS[name]
    bl = I.make_batch(spec, seed, dev)
    w = weights if weights is not None else I.make_layer_weights(spec, seed, 0, dev)
    if fold and w["ln1"] is not None:
        w = lb.folded_layer_weights(w)
    x, r = I.make_activations(spec, bl.num_tokens, seed, dev)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, dev)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    W = Workload()
    W.spec, W.bl, W.cfg, W.batch, W.w, W.x, W.r, W.kc, W.vc = spec, bl, cfg, batch, w, x, r, kc, vc
    W.hidden = x.clone()
    W.res_out = torch.empty_like(x)
    W.ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), dev)

    def step(stream=None):
        lb.layer_forward(cfg, w, batch, W.hidden, r, W.res_out, kc, vc, W.ws, stream=stream)

    W.step = step
    W.tokens_per_step = bl.num_tokens
    W.layers_n = 1
    return W


def layer_algorithmic(spec, bl):
    """Algorithmic bytes and flops of one layer step: every weight read once,
    KV read once per KV head, the new K/V written once, activations read or
    written once per materialised tensor; attention flops 4*d per visible
    (query, key, q-head) pair."""
    H, I, d, nq, nkv = spec.hidden, spec.intermediate, spec.head_dim, spec.n_heads, spec.n_kv_heads
    T = bl.num_tokens
    w_elems = (nq + 2 * nkv) * d * H + H * nq * d + 2 * I * H + H * I + 2 * H
    pairs = 0
    kv_read = 0
    for c, q in zip(bl.ctx_lens, bl.q_lens):
        kv_read += c + q
        for j in range(q):
            pairs += c + j + 1
    kv_bytes = kv_read * nkv * d * 2 * 2 + T * nkv * d * 2 * 2
    act_bytes = T * H * 2 * 2 * 3 + T * nq * d * 2 * 2 + T * I * 2 * 2 + T * 2 * I * 0
    flops = 2 * T * w_elems + 4 * d * pairs * nq
    return {"weight_bytes": w_elems * 2, "kv_bytes": kv_bytes, "act_bytes": act_bytes,
            "bytes": w_elems * 2 + kv_bytes + act_bytes, "flops": flops}


def time_steps(step, steps, warmup, world, sampler=None, counter=None):
    """Mean device time of one step in ms (max over ranks) and the clock record.
    counter: the library's launch counter; the kernels launched in the timed
    region are left in time_steps.launches."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
    n0 = counter() if counter else None
    e0.record(s)
    for _ in range(steps):
        step()
    e1.record(s)
    time_steps.launches = counter() - n0 if counter else None
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier(world)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(ms, world), clocks


def time_graph(step, steps, warmup, world):
    """Mean device time of one step replayed from a CUDA graph.  The step is
    run twice on a side stream first (every lazy set-up of the library happens
    outside the capture), captured once on that stream, then replayed on the
    current stream and timed like time_steps."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(stream=s)
    torch.cuda.synchronize()
    ms, _ = time_steps(g.replay, steps, warmup, world)
    del g
    return ms


def time_e2e(lb, W, steps, warmup, world, dev):
    """Same stack step through the public API with the step's inputs copied
    from pinned host memory and the sampled tokens copied back, every step.
    The inputs (token ids, positions, query_start_loc, seq_lens, block table:
    all int32) sit in one pinned host buffer and go over in one copy; the
    batch and the ids are views of the matching device buffer."""
    bl = W.bl
    parts = [("ids", W.ids), ("positions", bl.positions), ("qsl", bl.query_start_loc),
             ("seq_lens", bl.seq_lens), ("block_table", bl.block_table)]
    sizes = [t.numel() for _, t in parts]
    slots = [(n + 3) // 4 * 4 for n in sizes]  # each part starts on a 16-byte boundary
    host = torch.zeros(sum(slots), dtype=torch.int32).pin_memory()
    dev_buf = torch.empty(sum(slots), dtype=torch.int32, device=dev)
    views, off = {}, 0
    for (name, t), n, m in zip(parts, sizes, slots):
        host[off:off + n].copy_(t.reshape(-1).to(torch.int32).cpu())
        views[name] = dev_buf[off:off + n].view(t.shape)
        off += m
    out_host = torch.empty(bl.num_seqs, dtype=torch.int32).pin_memory()
    batch = lb.Batch(views["positions"], views["qsl"], views["seq_lens"], views["block_table"],
                     W.batch.num_blocks, W.batch.max_query_len, W.batch.max_seq_len)
    h2d = host.numel() * host.element_size()
    d2h = out_host.numel() * out_host.element_size()

    def step():
        dev_buf.copy_(host, non_blocking=True)
        W.step(batch=batch, ids=views["ids"])
        out_host.copy_(W.tokens, non_blocking=True)

    ms, _ = time_steps(step, steps, warmup, world)
    return ms, h2d, d2h


def time_kernel(fn, reps, warmup=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(reps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# --------------------------------------------------------------------------- CPU oracle sample


class OracleSample:
    """The CPU oracle on the first ``n_seqs`` decode sequences of the stack
    workload, through all layers, the final norm and lm_head.  Preparing the
    inputs (device->host copies, bf16->fp32 widening, compacting the sample's
    cache blocks) happens once, outside the timed calls."""

    def __init__(self, W, n_seqs=2, dtype=np.float32):
        from oracle import llama_oracle as O
        self.O, self.dtype = O, dtype
        spec, bl = W.spec, W.bl
        self.sh = O.LayerShape(spec.hidden, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.intermediate,
                               spec.rms_eps, spec.rope_theta, spec.rope_scaling, spec.block_size)
        qsl = bl.query_start_loc.cpu().numpy()
        seqs = list(range(n_seqs))
        rows = np.concatenate([np.arange(qsl[b], qsl[b + 1]) for b in seqs])
        bt_full = bl.block_table.cpu().numpy()
        nblk = [(bl.ctx_lens[b] + bl.q_lens[b] + 15) // 16 for b in seqs]
        used = np.concatenate([bt_full[b, :nblk[b]] for b in seqs]).astype(np.int64)
        bt = -np.ones((len(seqs), max(nblk)), np.int64)
        cur = 0
        for i in range(len(seqs)):
            bt[i, :nblk[i]] = np.arange(cur, cur + nblk[i])
            cur += nblk[i]
        q_lens = [bl.q_lens[b] for b in seqs]
        self.sqsl = np.concatenate([[0], np.cumsum(q_lens)])
        self.batch = O.Batch(bl.positions.cpu().numpy()[rows], self.sqsl, bl.seq_lens.cpu().numpy()[seqs], bt)
        used_t = torch.as_tensor(used, device=W.layers[0]["w_qkv"].device)

        def f(t):
            return t.float().cpu().numpy()

        def b16(t):
            return t.view(torch.int16).cpu().numpy().view(np.uint16)

        self.x0 = f(W.emb[W.ids[torch.as_tensor(rows, device=W.ids.device)].long()])
        self.layers = [O.LayerWeights(f(w["ln1"]), f(w["w_qkv"]), f(w["w_o"]), f(w["ln2"]), f(w["w_gate_up"]),
                                      f(w["w_down"])) for w in W.layers]
        self.caches = [(b16(kc.index_select(0, used_t)), b16(vc.index_select(0, used_t))) for kc, vc in W.caches]
        self.fn, self.lm = f(W.fn), f(W.lm)
        self.ntok = len(rows)
        self.ctx = [bl.ctx_lens[b] for b in seqs]

    def run(self):
        """One timed pass; returns the seconds spent inside oracle calls."""
        O, sh, dtype = self.O, self.sh, self.dtype
        x, r = self.x0, None
        elapsed = 0.0
        for ow, (kc, vc) in zip(self.layers, self.caches):
            kc, vc = kc.copy(), vc.copy()
            t0 = time.perf_counter()
            x, r = O.decoder_layer(sh, ow, self.batch, x, r, kc, vc, dtype=dtype)
            elapsed += time.perf_counter() - t0
        t0 = time.perf_counter()
        sel = O.last_token_rows(self.sqsl)
        hf, _ = O.fused_add_rms_norm(x[sel], r[sel], self.fn, sh.rms_eps, dtype)
        O.greedy_argmax(O.linear(hf, self.lm, dtype))
        return elapsed + time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- main


def run_ours(args, world, rank, local):
    from llama_decoder_layer_gb300 import binding as lb
    from llama_decoder_layer_gb300 import build as lbuild
    from llama_decoder_layer_gb300 import inputs as I

    lbuild.build()
    lb.lib()
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    seed = rank  # independent replicas: each rank its own sequences
    if args.workload == "gemm_gate_up":
        return run_gate_up(args, world, rank, local, lb, I, dev, peaks, peak_src)
    if args.workload in ("attn_prefill", "attn_decode"):
        return run_attention(args, world, rank, local, lb, I, dev, peaks, peak_src, seed)
    if args.workload != "stack_70b":
        return run_single_layer(args, world, rank, local, lb, I, dev, peaks, peak_src, seed)
    W = setup_stack(lb, I, seed, dev, fold=args.fold_norms)

    extra = {}
    if not args.no_extra:
        # Single-layer configurations, each timed as a workload of its own
        # before the stack: the 70B decode and prefill layers (weights of the
        # stack's layer 0, their own batches and caches) and the 8B decode
        # layer.  The decode layers go first: after a power-capped prefill
        # run the SM clock takes a while to come back, and the small decode
        # GEMMs are latency-bound.  Clocks are sampled over each timed region.
        for name in ("decode_70b", "decode_8b", "prefill_70b"):
            L = setup_layer(lb, I, name, seed, dev, weights=W.layers[0] if name != "decode_8b" else None,
                            fold=args.fold_norms)
            steps = max(args.steps, 30) if name.startswith("decode") else args.steps
            lms, lclocks = time_steps(L.step, steps, args.warmup, world, ClockSampler(local))
            alg = layer_algorithmic(L.spec, L.bl)
            tps = L.tokens_per_step * world / (lms / 1e3)
            extra[name] = {"tokens_per_s": round(tps, 1), "layer_ms": round(lms, 4),
                           "roofline": layer_roofline(name, alg, lms, peaks, peak_src), "clocks": lclocks}
            if name.startswith("decode"):
                gms = time_graph(L.step, steps, args.warmup, world)
                extra[name]["cuda_graph"] = {"layer_ms": round(gms, 4),
                                             "tokens_per_s": round(L.tokens_per_step * world / (gms / 1e3), 1),
                                             "roofline": layer_roofline(name, alg, gms, peaks, peak_src)}
            st, detail = lb.get_device_error()
            if st != lb.LLAMA_OK:
                raise RuntimeError(f"device error in {name}: {lb.status_string(st)}")
            del L
            torch.cuda.empty_cache()

    # main line: the stack step
    sampler = ClockSampler(local)
    ms, clocks = time_steps(W.step, args.steps, args.warmup, world, sampler, counter=lb.launch_count)
    stack_launches = time_steps.launches
    st, detail = lb.get_device_error()
    if st != lb.LLAMA_OK:
        raise RuntimeError(f"device error during the bench: {lb.status_string(st)} (detail {detail})")
    tok_layers = W.tokens_per_step * W.layers_n
    value = whole_job_rate(tok_layers, ms, world)

    # end to end through the public API with host buffers, right after the
    # device-side timing so both see the same thermal and power state
    e2e_ms, h2d, d2h = time_e2e(lb, W, args.steps, args.warmup, world, dev)
    e2e_value = tok_layers * world / (e2e_ms / 1e3)

    # dominant kernel: the gate_up GEMM with SiluAndMul.  Timed inside the stack
    # step: a pass of its own right after the timed region (the same thermal
    # state), with CUDA events around each of its launches in the layer loop
    # (llama_gate_up_timer_*); being part of a long step, it is compared with
    # the sustained peak.
    spec, T = W.spec, W.tokens_per_step
    W.step()
    torch.cuda.synchronize()
    lb.gate_up_timer_start(args.steps * W.layers_n)
    for _ in range(args.steps):
        W.step()
    torch.cuda.synchronize()
    tot_ms, n_timed = lb.gate_up_timer_stop()
    in_ms = tot_ms / max(n_timed, 1)
    # the same launch timed alone, for reference against the burst peak
    xin = I.normal_bf16((T, spec.hidden), 1.0, 0.0, 77, dev)
    aout = torch.empty((T, spec.intermediate), dtype=torch.bfloat16, device=dev)
    gws = lb.alloc_workspace(lb.linear_workspace_size(), dev)
    wgu = W.layers[0]["w_gate_up"]
    k_ms = time_kernel(lambda: lb.gate_up_silu(xin, wgu, aout, gws), reps=max(args.steps, 10))
    k_flops = 2.0 * T * 2 * spec.intermediate * spec.hidden
    in_tflops = k_flops / (in_ms / 1e3) / 1e12
    k_tflops = k_flops / (k_ms / 1e3) / 1e12
    roofline = {"kernel": "k_gemm_tc<SwiGLU> (gate_up_proj + SiluAndMul)", "bound": "tensor",
                "achieved": round(in_tflops, 1), "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": round(in_tflops / peaks["bf16_tflops_sustained"], 4),
                "peak_source": f"bf16_tflops_sustained ({peak_src}): the kernel is timed inside the stack step",
                "flops_per_launch": k_flops, "launch_ms": round(in_ms, 4), "launches_timed": n_timed,
                "traffic": GATE_UP_DRAM_BYTES_PER_LAUNCH,
                "alone": {"launch_ms": round(k_ms, 4), "achieved": round(k_tflops, 1), "peak": peaks["bf16_tflops"],
                          "frac": round(k_tflops / peaks["bf16_tflops"], 4),
                          "peak_source": f"bf16_tflops ({peak_src}, burst)"}}
    del xin, aout, gws


    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        osmp = OracleSample(W, n_seqs=2)
        secs = osmp.run()
        cpu = {"value": round(osmp.ntok * W.layers_n / secs, 4), "unit": "tokens/s per layer", "cores": cpu_cores(),
               "kind": "oracle", "seconds": round(secs, 2),
               "sample": f"{osmp.ntok} decode sequences (1 token each, contexts {osmp.ctx}) through all "
                         f"{W.layers_n} layers + final norm + lm_head, oracle in fp32 on the host"}
        del osmp

    # algorithmic totals of the stack step
    alg_layers = [layer_algorithmic(W.spec, W.bl) for _ in range(1)][0]
    stack_flops = alg_layers["flops"] * W.layers_n + 2.0 * W.bl.num_seqs * W.spec.hidden * W.spec.vocab
    tokens_per_step, layers_n = W.tokens_per_step, W.layers_n

    if not args.no_extra and not args.fold_norms:
        # the full-depth 80-layer decode step (193 GB on the device): the stack's buffers go first
        del W
        gc.collect()
        torch.cuda.empty_cache()
        r = deep_decode(args, world, rank, local, lb, I, dev, peaks, peak_src)
        B, L = r["B"], r["layers"]
        extra["decode_70b_80l"] = {
            "tokens_per_s_per_layer": round(B * L * world / (r["ms"] / 1e3), 1), "step_ms": round(r["ms"], 4),
            "roofline": r["roofline"],
            "clocks": r["clocks"],
            "cuda_graph": {"step_ms": round(r["graph_ms"], 4),
                           "tokens_per_s_per_layer": round(B * L * world / (r["graph_ms"] / 1e3), 1),
                           "roofline": r["graph_roofline"]},
            "config": f"embedding + {L} layers + final norm + lm_head + argmax, {B} decode seqs, ctx U[512,4096]"}
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(value, 1), "unit": "tokens/s per layer", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights of the 70B shape)",
        "config": {"workload": "stack_70b: 8 x 70B-shaped layers + final norm + lm_head(128256) + greedy argmax; "
                               "32 decode seqs (ctx U[1024,16384]) + 2 prefill chunks x 2048; 4128 tokens",
                   "tokens_per_step": tokens_per_step, "layers": layers_n,
                   "l2": "inputs larger than L2 (13.7 GB of weights per step)", "parallelism": f"replicas x{world}",
                   "norms": "folded into w_qkv / w_gate_up" if args.fold_norms else "separate"},
        "stack_tflops_per_s": round(stack_flops / (ms / 1e3) / 1e12, 1),
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s per layer", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": stack_launches,
        "cpu_baseline": cpu,
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)


def layer_roofline(name, alg, ms, peaks, peak_src):
    if name.startswith("decode") or name == "tiny":
        gbs = alg["bytes"] / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm_gbs ({peak_src})",
                "algorithmic_bytes": alg["bytes"], "traffic": None}
    tf = alg["flops"] / (ms / 1e3) / 1e12
    return {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
            "frac": round(tf / peaks["bf16_tflops_sustained"], 4),
            "peak_source": f"bf16_tflops_sustained ({peak_src})", "algorithmic_flops": alg["flops"], "traffic": None}


def run_gate_up(args, world, rank, local, lb, I, dev, peaks, peak_src):
    """The gate_up projection with its SiluAndMul epilogue alone, 70B weights,
    --gemm-tokens rows (4128, the stack's batch, by default: x 68 MB, W 940 MB,
    out 237 MB)."""
    spec = I.SPECS["stack_70b"]
    T = args.gemm_tokens
    x = I.normal_bf16((T, spec.hidden), 1.0, 0.0, 77, dev)
    w = I.normal_bf16((2 * spec.intermediate, spec.hidden), 0.02, 0.0, 78, dev)
    out = torch.empty((T, spec.intermediate), dtype=torch.bfloat16, device=dev)
    ws = lb.alloc_workspace(lb.linear_workspace_size(), dev)
    sampler = ClockSampler(local)
    ms, clocks = time_steps(lambda: lb.gate_up_silu(x, w, out, ws), args.steps, args.warmup, world, sampler,
                            counter=lb.launch_count)
    flops = 2.0 * T * 2 * spec.intermediate * spec.hidden
    tf = flops / (ms / 1e3) / 1e12
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(T * world / (ms / 1e3), 1), "unit": "tokens/s through gate_up_proj", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"gemm_gate_up: {T} x {2 * spec.intermediate} x {spec.hidden} + SiluAndMul",
                   "l2": "inputs larger than L2 (940 MB of weights)"},
        "roofline": {"kernel": "k_gemm_tc<SwiGLU>", "bound": "tensor", "achieved": round(tf, 1),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                     "peak_source": f"bf16_tflops ({peak_src}, burst)", "flops_per_launch": flops, "traffic": None},
        "clocks": clocks, "gpu_launches": time_steps.launches, "cpu_baseline": None, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_attention(args, world, rank, local, lb, I, dev, peaks, peak_src, seed):
    """The paged GQA attention of the 70B prefill (8 x 4096, causal) or decode
    (128 sequences, context U[512, 8192]) batch alone, q drawn N(0,1)."""
    spec = I.SPECS["prefill_70b" if args.workload == "attn_prefill" else "decode_70b"]
    bl = I.make_batch(spec, seed, dev)
    q = I.normal_bf16((bl.num_tokens, spec.n_heads, spec.head_dim), 1.0, 0.0, 5, dev)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, dev)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    out = torch.empty((bl.num_tokens, spec.n_heads * spec.head_dim), dtype=torch.bfloat16, device=dev)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, bl.num_tokens, bl.num_seqs, batch.max_seq_len), dev)
    sampler = ClockSampler(local)
    ms, clocks = time_steps(lambda: lb.paged_attention(cfg, batch, q, kc, vc, out, ws), args.steps, args.warmup,
                            world, sampler, counter=lb.launch_count)
    d, nq, nkv = spec.head_dim, spec.n_heads, spec.n_kv_heads
    pairs = sum(c * q_ + q_ * (q_ + 1) // 2 for c, q_ in zip(bl.ctx_lens, bl.q_lens))
    kv_bytes = sum(c + q_ for c, q_ in zip(bl.ctx_lens, bl.q_lens)) * nkv * d * 2 * 2
    io_bytes = bl.num_tokens * nq * d * 2 * 2
    if args.workload == "attn_prefill":
        tf = 4.0 * d * pairs * nq / (ms / 1e3) / 1e12
        roof = {"kernel": "k_attn_prefill", "bound": "tensor", "achieved": round(tf, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                "peak_source": f"bf16_tflops ({peak_src}, burst)", "traffic": None}
    else:
        gbs = (kv_bytes + io_bytes) / (ms / 1e3) / 1e9
        roof = {"kernel": "k_attn_decode + k_attn_combine", "bound": "hbm", "achieved": round(gbs, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                "peak_source": f"hbm_gbs ({peak_src})", "algorithmic_bytes": kv_bytes + io_bytes, "traffic": None}
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(bl.num_tokens * world / (ms / 1e3), 1), "unit": "tokens/s through attention",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload}, "roofline": roof, "clocks": clocks,
        "gpu_launches": time_steps.launches,
        "cpu_baseline": None, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_single_layer(args, world, rank, local, lb, I, dev, peaks, peak_src, seed):
    """One decoder layer of the named workload per step (residual in, residual out)."""
    L = setup_layer(lb, I, args.workload, seed, dev, fold=args.fold_norms)
    sampler = ClockSampler(local)
    ms, clocks = time_steps(L.step, args.steps, args.warmup, world, sampler, counter=lb.launch_count)
    st, detail = lb.get_device_error()
    if st != lb.LLAMA_OK:
        raise RuntimeError(f"device error during the bench: {lb.status_string(st)} (detail {detail})")
    alg = layer_algorithmic(L.spec, L.bl)
    value = L.tokens_per_step * world / (ms / 1e3)
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": args.workload, "tokens_per_step": L.tokens_per_step, "layers": 1,
                   "l2": "inputs larger than L2" if alg["bytes"] > L2_BYTES else "inputs smaller than L2",
                   "parallelism": f"replicas x{world}",
                   "norms": "folded into w_qkv / w_gate_up" if args.fold_norms else "separate"},
        "roofline": layer_roofline(args.workload, alg, ms, peaks, peak_src),
        "clocks": clocks, "gpu_launches": time_steps.launches, "cpu_baseline": None, "e2e": None,
    }
    if args.workload.startswith("decode"):
        # the same step replayed from a CUDA graph (launch overheads removed)
        gms = time_graph(L.step, args.steps, args.warmup, world)
        line["cuda_graph"] = {"ms_per_step": round(gms, 4),
                              "value": round(L.tokens_per_step * world / (gms / 1e3), 1),
                              "roofline": layer_roofline(args.workload, alg, gms, peaks, peak_src)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def deep_decode(args, world, rank, local, lb, I, dev, peaks, peak_src):
    """The full-depth 70B decode step: embedding, 80 layers, final norm,
    lm_head and greedy sampling in one llama_stack_forward call, timed eager
    and replayed from a CUDA graph.  Every layer has its own weight and cache
    buffers (137 GB + 48 GB); their values are layer 0's, copied, since
    drawing 68 G random numbers would dominate the run.  Returns the timing
    record (eager and graph, each with its HBM roofline)."""
    seed = 1000 + rank
    spec = I.SPECS["decode_70b_80l"]
    bl = I.make_batch(spec, seed, dev)
    w0 = I.make_layer_weights(spec, seed, 0, dev)
    layers = [w0] + [{k: v.clone() for k, v in w0.items()} for _ in range(spec.num_layers - 1)]
    kc0, vc0 = I.make_kv_cache(spec, bl.num_blocks, seed, 0, dev)
    caches = [(kc0, vc0)] + [(kc0.clone(), vc0.clone()) for _ in range(spec.num_layers - 1)]
    emb, ids, lm, fn = I.make_stack_extras(spec, bl.num_tokens, seed, dev)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    T, B = bl.num_tokens, bl.num_seqs
    hidden = torch.empty((T, spec.hidden), dtype=torch.bfloat16, device=dev)
    residual = torch.empty_like(hidden)
    tokens = torch.empty(B, dtype=torch.int32, device=dev)
    ws = lb.alloc_workspace(lb.workspace_size(cfg, T, B, batch.max_seq_len, spec.vocab), dev)
    kcs, vcs = [c[0] for c in caches], [c[1] for c in caches]

    def step(stream=None):
        lb.stack_forward(cfg, layers, fn, lm, batch, hidden, residual, kcs, vcs, tokens, ws, embed=emb,
                         input_ids=ids, stream=stream)

    sampler = ClockSampler(local)
    ms, clocks = time_steps(step, args.steps, args.warmup, world, sampler, counter=lb.launch_count)
    launches = time_steps.launches
    gms = time_graph(step, args.steps, args.warmup, world)
    st, detail = lb.get_device_error()
    if st != lb.LLAMA_OK:
        raise RuntimeError(f"device error in the 80-layer decode: {lb.status_string(st)} (detail {detail})")
    alg = layer_algorithmic(spec, bl)
    head_bytes = spec.vocab * spec.hidden * 2 + B * spec.vocab * 4
    step_bytes = spec.num_layers * alg["bytes"] + head_bytes

    def roof(t_ms):
        gbs = step_bytes / (t_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm_gbs ({peak_src})",
                "algorithmic_bytes": step_bytes, "traffic": None}

    rec = {"B": B, "T": T, "layers": spec.num_layers, "ms": ms, "graph_ms": gms, "clocks": clocks,
           "launches": launches, "step_bytes": step_bytes, "roofline": roof(ms), "graph_roofline": roof(gms)}
    del layers, caches, kcs, vcs, w0, kc0, vc0, emb, lm, ws
    torch.cuda.empty_cache()
    return rec


def run_deep_decode(args, world, rank, local):
    """--workload decode_70b_80l: the full-depth decode step as its own line."""
    from llama_decoder_layer_gb300 import binding as lb
    from llama_decoder_layer_gb300 import build as lbuild
    from llama_decoder_layer_gb300 import inputs as I
    lbuild.build()
    lb.lib()
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    r = deep_decode(args, world, rank, local, lb, I, dev, peaks, peak_src)
    B, L = r["B"], r["layers"]
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(B * L * world / (r["ms"] / 1e3), 1), "unit": "tokens/s per layer", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"], 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; every layer's buffers hold layer 0's random values)",
        "config": {"workload": f"decode_70b_80l: embedding + 80 x 70B-shaped layers + final norm + lm_head(128256) "
                               f"+ greedy argmax; {B} decode seqs, ctx U[512,4096]",
                   "tokens_per_step": r["T"], "layers": L,
                   "l2": f"inputs larger than L2 ({r['step_bytes'] / 1e9:.0f} GB per step)",
                   "parallelism": f"replicas x{world}"},
        "roofline": r["roofline"], "clocks": r["clocks"], "gpu_launches": r["launches"], "cpu_baseline": None,
        "e2e": None,
        "cuda_graph": {"ms_per_step": round(r["graph_ms"], 4),
                       "value": round(B * L * world / (r["graph_ms"] / 1e3), 1), "roofline": r["graph_roofline"]},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_sampler(args, world, rank, local):
    """llama_sample on the stack's head: 34 rows of fp32 logits over vocab
    128256, temperature 0.8, top-k 50, top-p 0.9, one uniform per row."""
    from llama_decoder_layer_gb300 import binding as lb
    from llama_decoder_layer_gb300 import build as lbuild
    lbuild.build()
    lb.lib()
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    rows, vocab = 34, 128256
    g = torch.Generator(device=dev)
    g.manual_seed(77 + rank)
    logits = torch.randn((rows, vocab), generator=g, device=dev) * 2.5
    temp = torch.full((rows,), 0.8, device=dev)
    top_k = torch.full((rows,), 50, dtype=torch.int32, device=dev)
    top_p = torch.full((rows,), 0.9, device=dev)
    u = torch.rand((rows,), generator=g, device=dev)
    tok = torch.empty(rows, dtype=torch.int32, device=dev)
    lp = torch.empty(rows, dtype=torch.float32, device=dev)
    sampler = ClockSampler(local)
    ms, clocks = time_steps(lambda: lb.sample(logits, temp, top_k, top_p, u, tok, lp), args.steps, args.warmup,
                            world, sampler, counter=lb.launch_count)
    nbytes = rows * vocab * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    # the same rows with no truncation (top-k off, top-p 1): the draw over the whole vocabulary
    top_k0 = torch.zeros_like(top_k)
    top_p1 = torch.ones_like(top_p)
    ms_full, _ = time_steps(lambda: lb.sample(logits, temp, top_k0, top_p1, u, tok, lp), args.steps, args.warmup,
                            world)
    # top-p alone (top-k off, top-p 0.9)
    ms_topp, _ = time_steps(lambda: lb.sample(logits, temp, top_k0, top_p, u, tok, lp), args.steps, args.warmup,
                            world)
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(rows * world / (ms / 1e3), 1), "unit": "sampled tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"sample: {rows} x {vocab} fp32 logits, temperature 0.8, top-k 50, top-p 0.9"},
        "roofline": {"kernel": "k_sample", "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm_gbs ({peak_src})",
                     "algorithmic_bytes": nbytes, "traffic": None,
                     "note": "a cluster of 4 CTAs per row, two passes over its 513 KB (top-k candidates, then the "
                             "selection in shared memory): latency-bound, not bandwidth-bound"},
        "clocks": clocks, "gpu_launches": time_steps.launches, "cpu_baseline": None, "e2e": None,
        "no_truncation": {"ms_per_step": round(ms_full, 4), "config": "temperature 0.8, top-k off, top-p 1"},
        "top_p_only": {"ms_per_step": round(ms_topp, 4), "config": "temperature 0.8, top-k off, top-p 0.9"},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_moe(args, world, rank, local):
    """The sparse MoE block (llama_moe_forward) on Qwen3-30B-A3B shapes: hidden
    2048, 128 experts, top-8, moe_intermediate 768, random-init weights.
    moe_decode: 64 tokens (HBM-bound: the experts the routing touches are read
    once); moe_prefill: 4096 tokens (311 GFLOP against 1.24 GB: on the ridge,
    the HBM time slightly the larger)."""
    from llama_decoder_layer_gb300 import binding as lb
    from llama_decoder_layer_gb300 import build as lbuild
    from llama_decoder_layer_gb300 import inputs as I
    lbuild.build()
    lb.lib()
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    H, E, K, Im = 2048, 128, 8, 768
    T = 64 if args.workload == "moe_decode" else 4096
    seed = 500 + rank
    h = I.normal_bf16((T, H), 1.0, 0.0, seed, dev)
    wr = I.normal_bf16((E, H), 0.02, 0.0, seed + 1, dev)
    w13 = I.normal_bf16((E, 2 * Im, H), 0.02, 0.0, seed + 2, dev)
    w2 = I.normal_bf16((E, H, Im), 0.02, 0.0, seed + 3, dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws = lb.alloc_workspace(lb.moe_workspace_size(H, E, K, Im, T), dev)
    lb.moe_forward(h, wr, w13, w2, K, out, ws, ids)
    torch.cuda.synchronize()
    touched = int(torch.unique(ids).numel())
    sampler = ClockSampler(local)
    ms, clocks = time_steps(lambda: lb.moe_forward(h, wr, w13, w2, K, out, ws), args.steps, args.warmup, world,
                            sampler, counter=lb.launch_count)
    st, detail = lb.get_device_error()
    if st != lb.LLAMA_OK:
        raise RuntimeError(f"device error during the bench: {lb.status_string(st)} (detail {detail})")
    flops = 2.0 * T * (E * H + K * (2 * Im * H + H * Im))
    nbytes = (E * H + touched * (2 * Im * H + H * Im)) * 2 + 2 * T * H * 2
    # the bound is whichever of the algorithmic bytes and flops takes longer at the measured peaks
    if nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12):
        gbs = nbytes / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm_gbs ({peak_src})",
                "algorithmic_bytes": nbytes, "experts_touched": touched, "traffic": None}
    else:
        tf = flops / (ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(tf / peaks["bf16_tflops"], 4), "peak_source": f"bf16_tflops ({peak_src}, burst)",
                "algorithmic_flops": flops, "traffic": None}
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(T * world / (ms / 1e3), 1), "unit": "tokens/s through the MoE block", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": f"{args.workload}: Qwen3-30B-A3B MoE block, {T} tokens, hidden {H}, {E} experts, "
                               f"top-{K}, moe_intermediate {Im}"},
        "roofline": roof, "clocks": clocks, "gpu_launches": time_steps.launches, "cpu_baseline": None, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_moe_layer(args, world, rank, local):
    """One Qwen3-30B-A3B MoE decoder layer (llama_moe_layer_forward) per step:
    qwen3_moe_decode = 64 decode sequences, contexts U[512, 4096];
    qwen3_moe_prefill = 4 prefill sequences x 2048 tokens."""
    import dataclasses
    from llama_decoder_layer_gb300 import binding as lb
    from llama_decoder_layer_gb300 import build as lbuild
    from llama_decoder_layer_gb300 import inputs as I
    lbuild.build()
    lb.lib()
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    seed = 600 + rank
    spec = I.SPECS[args.workload]
    E, K, Im = spec.extra["num_experts"], spec.extra["top_k"], spec.extra["moe_intermediate"]
    bl = I.make_batch(spec, seed, dev)
    w = I.make_moe_layer_weights(spec, seed, 0, dev)
    x, r = I.make_activations(spec, bl.num_tokens, seed, dev)
    kc, vc = I.make_kv_cache(spec, bl.num_blocks, seed, 0, dev)
    cfg = lb.LayerConfig.from_spec(spec)
    batch = lb.Batch.from_layout(bl)
    T = bl.num_tokens
    ws = lb.alloc_workspace(lb.moe_layer_workspace_size(cfg, E, K, Im, T, bl.num_seqs, batch.max_seq_len), dev)
    hid = x.clone()
    res = torch.empty_like(x)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    lb.moe_layer_forward(cfg, w, K, batch, hid, r, res, kc, vc, ws, ids)
    torch.cuda.synchronize()
    touched = int(torch.unique(ids).numel())

    def step():  # as the dense single-layer workloads: each step's input is the previous step's output
        lb.moe_layer_forward(cfg, w, K, batch, hid, r, res, kc, vc, ws)

    sampler = ClockSampler(local)
    ms, clocks = time_steps(step, args.steps, args.warmup, world, sampler, counter=lb.launch_count)
    st, detail = lb.get_device_error()
    if st != lb.LLAMA_OK:
        raise RuntimeError(f"device error during the bench: {lb.status_string(st)} (detail {detail})")
    H = spec.hidden
    alg = layer_algorithmic(dataclasses.replace(spec, intermediate=0), bl)  # norms, attention, o_proj
    moe_bytes = (E * H + touched * 3 * Im * H) * 2
    nbytes = alg["bytes"] + moe_bytes
    flops = alg["flops"] + 2 * T * (E * H + K * 3 * Im * H)
    if nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops_sustained"] * 1e12):
        gbs = nbytes / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"hbm_gbs ({peak_src})",
                "algorithmic_bytes": nbytes, "experts_touched": touched, "traffic": None}
    else:
        tf = flops / (ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops_sustained"], 4),
                "peak_source": f"bf16_tflops_sustained ({peak_src})", "algorithmic_flops": flops, "traffic": None}
    line = {
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(T * world / (ms / 1e3), 1), "unit": "tokens/s per Qwen3-MoE layer", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": f"{args.workload}: one Qwen3-30B-A3B MoE decoder layer (hidden 2048, 32/4 heads, "
                               f"128 experts, top-8, moe_intermediate 768), {T} tokens in {bl.num_seqs} sequences",
                   "tokens_per_step": T, "layers": 1},
        "roofline": roof, "clocks": clocks, "gpu_launches": time_steps.launches, "cpu_baseline": None, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    """Times the CPU oracle (fp32) on a bounded sample of the stack workload:
    each step runs one decode sequence through all layers + head."""
    if rank != 0:
        return
    from llama_decoder_layer_gb300 import inputs as I
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    # inputs come from the seeded generator (device only holds them; no kernel of this library runs)
    import types
    spec = I.SPECS["stack_70b"]
    bl = I.make_batch(spec, 0, dev)
    W = types.SimpleNamespace(spec=spec, bl=bl, layers_n=spec.num_layers)
    W.layers = [I.make_layer_weights(spec, 0, l, dev) for l in range(spec.num_layers)]
    W.emb, W.ids, W.lm, W.fn = I.make_stack_extras(spec, bl.num_tokens, 0, dev)
    W.caches = [I.make_kv_cache(spec, bl.num_blocks, 0, l, dev) for l in range(spec.num_layers)]
    W.hidden = W.emb
    osmp = OracleSample(W, n_seqs=1)
    del W.layers, W.caches, W.emb, W.lm
    times = []
    for i in range(args.warmup + args.steps):
        secs = osmp.run()
        if i >= args.warmup:
            times.append(secs)
    total = sum(times)
    value = osmp.ntok * W.layers_n * len(times) / total
    line = {
        "impl": "reference",
        "metric": "tokens/s per 70B-shape decoder layer (decode, prefill) & % of HBM/TC roofline",
        "value": round(value, 4), "unit": "tokens/s per layer", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "stack_70b (sample: 1 decode sequence through 8 layers + final norm + lm_head)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s per layer", "cores": cpu_cores(),
                         "kind": "oracle", "sample": "1 decode sequence per step through all 8 layers + head, fp32"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s per layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stack_70b",
                    choices=["stack_70b", "decode_70b", "prefill_70b", "decode_8b", "tiny", "gemm_gate_up",
                             "attn_prefill", "attn_decode", "decode_70b_80l", "sample", "moe_decode",
                             "moe_prefill", "qwen3_moe_decode", "qwen3_moe_prefill"],
                    help="stack_70b (default), one single-layer workload, or gemm_gate_up: the stack's "
                         "dominant kernel alone (4128 x 57344 x 8192, for profiling); attn_prefill / "
                         "attn_decode: the paged attention of the 70B prefill / decode batch alone; "
                         "decode_70b_80l: the full-depth 70B decode step (~193 GB on the device); sample: "
                         "llama_sample on the stack's 34 x 128256 head; moe_decode / moe_prefill: the "
                         "Qwen3-30B-A3B MoE block over 64 / 4096 tokens; qwen3_moe_decode / qwen3_moe_prefill: "
                         "one Qwen3-30B-A3B MoE decoder layer, 64 decode sequences / 4 x 2048 prefill")
    ap.add_argument("--gemm-tokens", type=int, default=4128, help="rows of the gemm_gate_up workload")
    ap.add_argument("--no-extra", action="store_true", help="skip the single-layer decode/prefill results")
    ap.add_argument("--fold-norms", action="store_true",
                    help="run the layers with the RMSNorm weights folded into w_qkv / w_gate_up")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload == "decode_70b_80l":
        run_deep_decode(args, world, rank, local)
    elif args.workload == "sample":
        run_sampler(args, world, rank, local)
    elif args.workload in ("moe_decode", "moe_prefill"):
        run_moe(args, world, rank, local)
    elif args.workload in ("qwen3_moe_decode", "qwen3_moe_prefill"):
        run_moe_layer(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
