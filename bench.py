#!/usr/bin/env python
"""Benchmark: verified draft-tree nodes per second for one token-tree verification step.

One step = one spec_tree_attention call (tree-masked attention of the draft tree over its KV
prefix, one layer) + one spec_tree_verify call (speculative-sampling accept/reject, walk, bonus
draw) on one batch of the workload.  Default workload: the EAGLE static tree on a Vicuna-7B
attention shape (batch 1, 32 heads x 128, prefix 1024, 60-node tree of depth 6 / width <= 10,
vocabulary 32000, temperature 1.0), seeded synthetic data.

Timing: W warm-up steps, then exactly K steps replayed from CUDA graphs (one step per rotated copy
of the inputs; the copies together exceed twice the L2 size, so every step reads HBM), bracketed by
a barrier and torch.cuda.synchronize(); CUDA events on the launching stream.  With torchrun (N > 1)
every rank runs an independent replica (the step has no cross-GPU exchange); rank 0 prints one JSON
line with value = all ranks' nodes / max-over-ranks time.

--impl reference times the CPU oracle (fp64 NumPy, one thread) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified tree nodes/sec (attn+verify) at 1 GB300 and % of HBM roofline"
UNIT = "nodes/s"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="eagle_vicuna7b")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the configuration's batch (e.g. a smaller case to profile)")
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true",
                    help="skip the paged-attention and KV-compaction measurements")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (batched GQA, long context, stress sweep, T=0)")
    ap.add_argument("--cpu-child", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------------
# workload and algorithmic bytes
# ------------------------------------------------------------------------------------------------
def make_inputs(cfg_name, T, seed, batch=None):
    from speculative_decoding_token_spec_gb300 import workloads as W
    cfg = W.config(cfg_name) if batch is None else W.config(cfg_name, B=batch)
    ac = W.make_attention_case(cfg, seed=seed)
    vc = W.make_verify_case(cfg, T, seed=seed)
    return cfg, ac, vc


def workload_name(cfg, T):
    """The workload string both arms print: configuration, shapes, prefix, tree, vocabulary, T."""
    pre = (f"prefix={cfg.prefix[1]}" if cfg.prefix[0] == "fixed"
           else f"prefix=U[{cfg.prefix[1]},{cfg.prefix[2]}]")
    return (f"{cfg.name}: B={cfg.B} Hq={cfg.Hq} Hkv={cfg.Hkv} D={cfg.D} {pre} N={cfg.N} "
            f"V={cfg.V} T={T}")


def algorithmic_bytes(cfg, ac, vc):
    """Bytes the step must move at minimum.

    attention: K and V of every visible slot (prefix + tree) per KV head, Q in, O out, LSE out.
    verify: the target-logit row of every internal node (4V each) plus the terminal row of target
    logits and draft probabilities (8V) per sequence.
    """
    import numpy as np
    B, N, Hq, Hkv, D = ac.shape
    kv = sum(int(Hkv) * (int(L) + N) * D * 2 * 2 for L in ac.prefix_lens)
    qo = 2 * B * N * Hq * D * 2
    attn = kv + qo + B * Hq * N * 4
    V = vc.target_logits.shape[2]
    internal = 0
    for b in range(B):
        internal += len(np.unique(vc.tree_parent[b, 1:]))
    verify = internal * 4 * V + B * 8 * V
    flops = sum(4 * Hq * N * (int(L) + N) * D for L in ac.prefix_lens)
    return attn, verify, flops


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def _once(self):
        try:
            r = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}", "-i", str(self.index),
                                "--format=csv,noheader,nounits"], capture_output=True, text=True,
                               timeout=10)
            return [l for l in r.stdout.splitlines() if l.strip()]
        except Exception:
            return []

    def start(self):
        self.lines += self._once()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "-i", str(self.index),
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=10)
                self.lines += [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()
        self.lines += self._once()
        return self.summary()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (a child process: fresh interpreter, one BLAS thread)
# ------------------------------------------------------------------------------------------------
def cpu_oracle_child(spec):
    """Times the fp64 oracle on a bounded sample of the workload; prints one JSON object."""
    import numpy as np
    from oracle import attention as OA
    from oracle import verify as OV
    from speculative_decoding_token_spec_gb300 import workloads as W
    cfg_name, T, seed, steps, budget, threads, fixed = spec.split(":")
    T, seed, steps, budget, threads = float(T), int(seed), int(steps), float(budget), int(threads)
    fixed = int(fixed)
    cfg, ac, vc = make_inputs(cfg_name, T, seed)
    B, N = ac.q.shape[:2]
    q = W.bf16_to_f64(ac.q)
    k = W.bf16_to_f64(ac.k_cache)
    v = W.bf16_to_f64(ac.v_cache)

    def one(nodes):
        OA.tree_attention(q, k, v, ac.prefix_lens, ac.tree_parent, ac.scale, nodes=nodes)
        OV.tree_verify(vc.target_logits, vc.draft_probs, vc.tree_tokens, vc.tree_parent,
                       vc.uniforms, T)

    # size the per-step sample: all nodes if the budget allows, else fewer attention nodes
    t0 = time.perf_counter()
    one([(0, 0)])
    t_min = time.perf_counter() - t0
    t0 = time.perf_counter()
    OA.tree_attention(q, k, v, ac.prefix_lens, ac.tree_parent, ac.scale,
                      nodes=[(b, i) for b in range(B) for i in range(min(N, 4))])
    t_node = (time.perf_counter() - t0) / (B * min(N, 4))
    per_step = budget / max(steps, 1)
    n_nodes = int(max(1, min(B * N, (per_step - t_min) / max(t_node, 1e-9) + 1)))
    if fixed > 0:  # the same sample as another run of this leg
        n_nodes = min(fixed, B * N)
    all_nodes = [(b, i) for b in range(B) for i in range(N)]
    sample = all_nodes[:n_nodes]
    t0 = time.perf_counter()
    for _ in range(steps):
        one(sample)
    dt = time.perf_counter() - t0
    print(json.dumps({"value": n_nodes * steps / dt, "steps": steps, "nodes_per_step": n_nodes,
                      "seconds": dt, "cores": threads,
                      "sample": f"{steps} oracle step(s) of {cfg_name}: attention for {n_nodes} of "
                                f"{B * N} nodes (all heads) + full-tree verification at T={T}"}))


def run_cpu_oracle(cfg_name, T, seed, steps, budget, threads=1, n_nodes=0):
    """The oracle in a child process whose BLAS / OpenMP pools hold `threads` threads; with
    n_nodes > 0 the sample is that many attention nodes (else sized by the budget)."""
    n = str(int(threads))
    env = dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n,
               CUDA_VISIBLE_DEVICES="")
    spec = f"{cfg_name}:{T}:{seed}:{steps}:{budget}:{n}:{int(n_nodes)}"
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", spec],
                       capture_output=True, text=True, env=env, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError(f"cpu oracle child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for l in f:
                if l.lower().startswith(("model name", "cpu part", "hardware")):
                    return l.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


# ------------------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ------------------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def combine_ranks(total_ms, units, device):
    """The job's aggregate over ranks: the longest timed region (max) and the units every rank
    processed (sum).  Identity without an initialised process group of more than one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(total_ms), float(units)
    import torch
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(u)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch
    import speculative_decoding_token_spec_gb300 as st

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    cfg, ac, vc = make_inputs(args.config, args.temperature, args.seed, args.batch)
    B, N, Hq, Hkv, D = ac.shape
    V = vc.target_logits.shape[2]
    T = args.temperature
    attn_bytes, verify_bytes, attn_flops = algorithmic_bytes(cfg, ac, vc)
    hbm_gbs, tc_tflops, peak_src = peaks()
    L2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def to_dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        return t.view(dtype) if dtype is not None else t

    host_inputs = {
        "q": ac.q, "k": ac.k_cache, "v": ac.v_cache, "lens": ac.prefix_lens,
        "parent": ac.tree_parent, "logits": vc.target_logits, "probs": vc.draft_probs,
        "tokens": vc.tree_tokens, "unif": vc.uniforms,
    }
    per_copy = sum(a.nbytes for a in host_inputs.values())
    copies = max(2, math.ceil(2 * L2 / per_copy))
    ws_attn = st.spec_tree_attention_workspace(B, N, Hq, Hkv, D, ac.Lmax)
    ws_ver = st.spec_tree_verify_workspace(B, N, V)

    def make_copy():
        c = {k: to_dev(a, torch.bfloat16 if k in ("q", "k", "v") else None)
             for k, a in host_inputs.items()}
        c["out"] = torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev)
        c["lse"] = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
        c["ws_a"] = torch.empty((max(ws_attn, 16),), dtype=torch.uint8, device=dev)
        c["ws_v"] = torch.empty((max(ws_ver, 16),), dtype=torch.uint8, device=dev)
        c["st_a"] = torch.zeros((B,), dtype=torch.int32, device=dev)
        c["st_v"] = torch.zeros((B,), dtype=torch.int32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        c["vout"] = {"accept_len": torch.empty((B,), **i32),
                     "accepted_tokens": torch.empty((B, N), **i32),
                     "bonus": torch.empty((B,), **i32),
                     "accepted_nodes": torch.empty((B, N), **i32)}
        return c

    bufs = [make_copy() for _ in range(copies)]

    def attn(c):
        st.spec_tree_attention(c["q"], c["k"], c["v"], c["lens"], c["parent"],
                               softmax_scale=ac.scale, out=c["out"], out_lse=c["lse"],
                               workspace=c["ws_a"], status=c["st_a"])

    def verify(c):
        st.spec_tree_verify(c["logits"], c["probs"] if T > 0 else None, c["tokens"], c["parent"],
                            c["unif"], T, outputs=c["vout"], workspace=c["ws_v"],
                            status=c["st_v"])

    def step(c):
        attn(c)
        verify(c)

    launches_per_step = 2  # one tree-attention kernel, one verification kernel

    # warm-up (eager), also validates the call path
    torch.cuda.nvtx.range_push("warm-up")
    for i in range(max(args.warmup, 3)):
        step(bufs[i % copies])
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    assert int(bufs[0]["st_a"].sum()) == 0 and int(bufs[0]["st_v"].sum()) == 0, "status"

    # CUDA graphs: one step per rotated copy, nothing between the kernels (so each launch can
    # overlap the previous kernel's tail through programmatic dependent launch)
    K = args.steps
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    fn(bufs[i])
        return g

    g_full = capture(step, copies)
    rem = K % copies
    g_rem = capture(step, rem) if rem else None
    g_attn, g_ver = capture(attn, copies), capture(verify, copies)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):  # first replays upload the graphs: keep them out of every timed region
        for g in (g_full, g_rem, g_attn, g_ver):
            if g is not None:
                g.replay()
    torch.cuda.synchronize()

    def timed(fn, name="timed region"):
        """CUDA-event time of fn() (ms), inside an NVTX range named `name` for profiler timelines."""
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push(name)
        a0.record()
        fn()
        a1.record()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        barrier()
        return a0.elapsed_time(a1)

    # ---- timed region: K steps
    props = torch.cuda.get_device_properties(dev)
    clocks = ClockSampler(getattr(props, "uuid", None) and f"GPU-{props.uuid}" or local)
    clocks.start()

    def run_steps():
        for _ in range(K // copies):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()

    total_ms = timed(run_steps, "steps: attention + verification")
    # ---- per-call timed regions: the same rotated copies, one kernel kind per graph
    reps = max(1, -(-300 // copies))  # about 300 calls per region, whatever --steps is
    attn_ms = timed(lambda: [g_attn.replay() for _ in range(reps)],
                    "per call: spec_tree_attention") / (reps * copies)
    ver_ms = timed(lambda: [g_ver.replay() for _ in range(reps)],
                   "per call: spec_tree_verify") / (reps * copies)
    clk = clocks.stop()
    per_call = (f"separate timed regions of {reps * copies} calls each, replaying graphs of one call "
                "over the rotated copies (back-to-back launches of that kernel)")

    # max over ranks, sum of units
    total_ms, units = combine_ranks(total_ms, B * N * K, dev)
    value = units / (total_ms / 1e3)
    ms_per_step = total_ms / K

    # ---- end to end through the public API with host buffers (pinned), copies in the region
    e2e = None
    if not args.no_e2e:
        pinned = {k: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                  for k, a in host_inputs.items()}
        res_host = {"out": torch.empty((B, N, Hq, D), dtype=torch.bfloat16).pin_memory(),
                    "accept_len": torch.empty((B,), dtype=torch.int32).pin_memory(),
                    "accepted_tokens": torch.empty((B, N), dtype=torch.int32).pin_memory(),
                    "bonus": torch.empty((B,), dtype=torch.int32).pin_memory()}
        h2d = sum(p.numel() * p.element_size() for p in pinned.values())
        d2h = sum(p.numel() * p.element_size() for p in res_host.values())
        K2 = min(K, 1000)
        # Pipelined over two device buffer sets: step k copies its inputs into set k % 2 on two
        # copy streams (the inputs split by bytes), once the step that last read that set is done;
        # its calls wait for those copies; its results come back on the compute stream.
        main = torch.cuda.current_stream()
        cstreams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
        order = sorted(pinned, key=lambda k: -pinned[k].numel() * pinned[k].element_size())
        lanes, load = ([], []), [0, 0]
        for k in order:  # largest first onto the less loaded stream
            i = 0 if load[0] <= load[1] else 1
            lanes[i].append(k)
            load[i] += pinned[k].numel() * pinned[k].element_size()
        sets = [bufs[0], bufs[1]]
        freed = [None, None]  # event: the last step on set i is done with its inputs

        def e2e_step(k):
            c = sets[k % 2]
            ready = []
            for i, cs in enumerate(cstreams):
                if freed[k % 2] is not None:
                    cs.wait_event(freed[k % 2])
                with torch.cuda.stream(cs):
                    for name in lanes[i]:
                        dst = c[name].view(torch.uint16) if name in ("q", "k", "v") else c[name]
                        dst.copy_(pinned[name], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                    ready.append(ev)
            for ev in ready:
                main.wait_event(ev)
            step(c)
            done = torch.cuda.Event()
            done.record(main)
            freed[k % 2] = done
            res_host["out"].copy_(c["out"], non_blocking=True)
            for name in ("accept_len", "accepted_tokens", "bonus"):
                res_host[name].copy_(c["vout"][name], non_blocking=True)

        for k in range(4):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for cs in cstreams:  # nothing of the timed steps starts before e0
            cs.wait_event(e0)
        for k in range(K2):
            e2e_step(k)
        for cs in cstreams:
            main.wait_stream(cs)
        e1.record()
        torch.cuda.synchronize()
        barrier()
        e_ms, e_units = combine_ranks(e0.elapsed_time(e1), B * N * K2, dev)
        e2e = {"value": e_units / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": K2,
               "note": "per step: pinned host inputs copied in (two copy streams, two device "
                       "buffer sets, so step k+1's copies overlap step k's calls), C-ABI calls, "
                       "results copied out"}

    if rank != 0:
        return
    # the other workloads' CPU legs (spawned workers) overlap the GPU work from here on; started
    # earlier, their input generation and fp64 oracle compete with the e2e region's copies for the
    # host's memory bandwidth (e2e 150 K against 320 K nodes/s measured)
    pool, futs = (None, None)
    if not args.no_configs and ws == 1:
        pool, futs = start_cpu_legs(args.seed)
    nxt = None if args.no_next else measure_next_rows(args, cfg, bufs, attn_bytes, hbm_gbs,
                                                      attn_ms, timed, dev, L2, tc_tflops)
    others = None
    if futs is not None:
        others = measure_other_workloads(args, dev, futs, hbm_gbs, tc_tflops, timed, L2)
        pool.shutdown()
    # ---- CPU oracle baseline (bounded sample)
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        try:
            r = run_cpu_oracle(args.config, T, args.seed, steps=50, budget=20.0)
            cpu = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                   "sample": r["sample"], "cpu": cpu_model(),
                   "nodes_per_step": r["nodes_per_step"]}
        except Exception as exc:  # pragma: no cover
            cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"failed: {exc}"}
    # the same oracle with every host core in its BLAS / OpenMP pools (a shorter sample)
    cpu_all = None
    if not args.no_cpu_baseline and ws == 1:
        ncores = (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                  else (os.cpu_count() or 1))
        if ncores > 1:
            try:
                n1 = (cpu or {}).get("nodes_per_step") or 0
                r = run_cpu_oracle(args.config, T, args.seed, steps=50, budget=10.0,
                                   threads=ncores, n_nodes=n1)
                cpu_all = {"value": r["value"], "unit": UNIT, "cores": r["cores"],
                           "kind": "oracle", "sample": r["sample"]}
            except Exception as exc:  # pragma: no cover
                cpu_all = {"value": None, "unit": UNIT, "cores": ncores, "kind": "oracle",
                           "sample": f"failed: {exc}"}

    attn_gbs = attn_bytes / (attn_ms * 1e-3) / 1e9
    ver_gbs = verify_bytes / (ver_ms * 1e-3) / 1e9
    # large problems verify along the accepted path only: the rows that form reads
    path_form = B * N * V * 4 > (64 << 20)
    path_bytes = None
    if path_form:
        out0 = bufs[0]["vout"]
        lens = out0["accept_len"].cpu().numpy()
        nodes = out0["accepted_nodes"].cpu().numpy()
        par0 = vc.tree_parent
        path_bytes = 0
        for b in range(B):
            for j in [0] + [int(x) for x in nodes[b, :max(int(lens[b]), 0)]]:
                has_kids = bool((par0[b, 1:] == j).any())
                path_bytes += 4 * V * (2 if (T > 0 and has_kids) else 1)
    step_roof_s = (attn_bytes + verify_bytes) / (hbm_gbs * 1e9)
    traffic = profiled_traffic("tree_attn")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the EAGLE static-tree workload, no datasets)",
        "config": {"workload": workload_name(cfg, T),
                   "batch": B, "tree_nodes": N, "vocab": V, "temperature": T,
                   "l2": f"inputs rotated over {copies} device copies "
                         f"({copies * per_copy / 2**20:.0f} MiB > 2x L2 {L2 / 2**20:.0f} MiB)",
                   "graphs": "one CUDA graph per rotation of copies",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "kernel": "tree_attn_kernel (split-KV, splits combined in the cluster)",
                     "achieved": attn_gbs, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": attn_gbs / hbm_gbs, "traffic": traffic,
                     "algorithmic_bytes": attn_bytes, "avg_launch_us": attn_ms * 1e3,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"},
        "step": {"attn_us": attn_ms * 1e3, "verify_us": ver_ms * 1e3,
                 "verify_gbs": ver_gbs, "attn_bytes": attn_bytes, "verify_bytes": verify_bytes,
                 "verify_form": "path only (one cluster per sequence)" if path_form
                                else "every node at once",
                 "verify_read_bytes": path_bytes,
                 "verify_read_gbs": (path_bytes / (ver_ms * 1e-3) / 1e9) if path_bytes else None,
                 "attn_tflops": attn_flops / (attn_ms * 1e-3) / 1e12,
                 "hbm_roofline_frac": step_roof_s / (ms_per_step * 1e-3),
                 "roofline_note": "T_roof = (attn + verify algorithmic bytes) / measured HBM GB/s; "
                                  "frac = T_roof / ms_per_step",
                 "per_call_timing": per_call},
        "clocks": clk,
        "gpu_launches": launches_per_step * K,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "next_rows": nxt,
        "configs": others,
    }
    print(json.dumps(line))


def measure_next_rows(args, cfg, bufs, attn_bytes, hbm_gbs, attn_ms, timed, dev, L2,
                      tc_tflops):
    """Paged-cache attention (16-slot pages), post-accept KV compaction, filtered verification,
    dynamic tree construction and the fused LM head on this workload.

    Paged attention: the same queries, tree and prefix over pages in a random physical order,
    rotated over device copies larger than 2 x L2, timed per call from CUDA graphs; its
    algorithmic bytes are those of the contiguous call.  Compaction: the accepted paths that the
    verification kernel produced in this run, applied to each copy's contiguous cache (in place,
    after every other measurement), timed the same way; algorithmic bytes = the moved rows read
    and written.
    """
    import numpy as np
    import torch
    import speculative_decoding_token_spec_gb300 as st
    from speculative_decoding_token_spec_gb300 import workloads as W
    page = 16
    pc = W.make_paged_attention_case(cfg, page, seed=args.seed)
    per_copy = pc.k_pages.nbytes * 2 + pc.q.nbytes
    ncp = max(2, math.ceil(2 * L2 / per_copy))
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    pcs = [{"q": to_dev(pc.q).view(torch.bfloat16), "k": to_dev(pc.k_pages).view(torch.bfloat16),
            "v": to_dev(pc.v_pages).view(torch.bfloat16), "t": to_dev(pc.block_table),
            "lens": to_dev(pc.prefix_lens), "par": to_dev(pc.tree_parent),
            "out": torch.empty(pc.q.shape, dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((pc.q.shape[0], pc.q.shape[2], pc.q.shape[1]),
                               dtype=torch.float32, device=dev),
            "st": torch.zeros((pc.q.shape[0],), dtype=torch.int32, device=dev)}
           for _ in range(ncp)]

    def paged(c):
        st.spec_tree_attention_paged(c["q"], c["k"], c["v"], c["t"], c["lens"], c["par"],
                                     softmax_scale=pc.scale, out=c["out"], out_lse=c["lse"],
                                     status=c["st"])

    def compact(c):
        st.spec_kv_compact(c["k"], c["v"], c["lens"], c["vout"]["accept_len"],
                           c["vout"]["accepted_nodes"], new_prefix_lens=c["new_lens"],
                           status=c["st_c"])

    for c in bufs:
        c["new_lens"] = torch.empty_like(c["lens"])
        c["st_c"] = torch.zeros_like(c["lens"])
    for _ in range(3):
        for c in pcs:
            paged(c)
        for c in bufs:
            compact(c)
    torch.cuda.synchronize()
    assert all(int(c["st"].sum()) == 0 for c in pcs) and all(int(c["st_c"].sum()) == 0 for c in bufs)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())

    def capture(fn, items):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for c in items:
                    fn(c)
        return g

    # filtered verification (top-k 50, top-p 0.9) on the same rotated copies as verification
    B, N, V = bufs[0]["logits"].shape
    T = args.temperature if args.temperature > 0 else 1.0
    top_k, top_p = 50, 0.9
    ws_f = st.spec_tree_verify_filtered_workspace(B, N, V)
    for c in bufs:
        c["ws_f"] = torch.empty((ws_f,), dtype=torch.uint8, device=dev)
        c["st_f"] = torch.zeros_like(c["lens"])
        c["fout"] = {k: torch.empty_like(v) for k, v in c["vout"].items()}

    def filtered(c):
        st.spec_tree_verify_filtered(c["logits"], c["probs"], c["tokens"], c["parent"],
                                     c["unif"], T, top_k=top_k, top_p=top_p, outputs=c["fout"],
                                     workspace=c["ws_f"], status=c["st_f"])

    def plain(c):
        st.spec_tree_verify(c["logits"], c["probs"], c["tokens"], c["parent"], c["unif"], T,
                            outputs=c["fout"], workspace=c["ws_f"], status=c["st_f"])

    for _ in range(3):
        for c in bufs:
            filtered(c)
    torch.cuda.synchronize()
    assert all(int(c["st_f"].sum()) == 0 for c in bufs)

    # dynamic tree construction: K = 10 candidates per expanded node, depth 6, this workload's
    # vocabulary and tree size, rows rotated over copies larger than 2 x L2
    tK, tD = 10, 6
    tcase = W.make_tree_build_case(B, tK, tD, V, seed=args.seed)
    ncp_t = max(2, math.ceil(2 * L2 / tcase.draft_rows.nbytes))
    ws_t = st.spec_tree_build_workspace(B, tK, tD)
    i32 = dict(dtype=torch.int32, device=dev)
    tcs = [{"levels": [to_dev(tcase.level_rows(d)) for d in range(1, tD + 1)],
            "roots": to_dev(tcase.root_tokens), "ws": torch.empty((ws_t,), dtype=torch.uint8,
                                                                 device=dev),
            "ft": torch.empty((B, tK), **i32), "fs": torch.empty((B, tK), **i32),
            "st": torch.zeros((B,), **i32),
            "out": {k: torch.empty((B, N), **i32) for k in ("tree_tokens", "tree_parent",
                                                            "node_row")}}
           for _ in range(ncp_t)]
    for c in tcs:
        c["out"]["node_value"] = torch.empty((B, N), dtype=torch.float32, device=dev)

    def expand_all(c):
        for d in range(1, tD + 1):
            st.spec_tree_expand(c["levels"][d - 1], tK, tD, d, c["ws"], frontier_tokens=c["ft"],
                                frontier_parent_slot=c["fs"], status=c["st"])

    def finalize(c):
        st.spec_tree_finalize(c["ws"], c["roots"], tK, tD, N, outputs=c["out"], status=c["st"])

    def build(c):
        expand_all(c)
        finalize(c)

    for _ in range(3):
        for c in tcs:
            build(c)
    torch.cuda.synchronize()
    assert all(int(c["st"].sum()) == 0 for c in tcs)

    # fused LM head: hidden [B N, H] (H = Hq D of this workload) times the head [V, H], reduced to
    # the verification statistics; the head alone is larger than 2 x L2, so every call reads HBM
    lm_h = cfg.Hq * cfg.D
    lm_m = B * N
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 17)
    lm_w = (torch.randn((V, lm_h), generator=gen, device=dev)
            * (3.0 / math.sqrt(lm_h))).to(torch.bfloat16)
    lm_x = torch.randn((lm_m, lm_h), generator=gen, device=dev).to(torch.bfloat16)
    lm_out = {"max": torch.empty((lm_m,), dtype=torch.float32, device=dev),
              "sumexp": torch.empty((lm_m,), dtype=torch.float32, device=dev),
              "argmax": torch.empty((lm_m,), dtype=torch.int32, device=dev)}
    lm_ws = torch.empty((st.spec_lm_head_stats_workspace(lm_m, V),), dtype=torch.uint8,
                        device=dev)
    lm_st = torch.zeros((1,), dtype=torch.int32, device=dev)

    lm_p = st.spec_lm_head_pack(lm_w)  # the head in tile-major order, made once

    def lmhead(_c=None):
        st.spec_lm_head_stats(lm_x, lm_p, T, outputs=lm_out, workspace=lm_ws, status=lm_st,
                              packed_vocab=V)

    def lmhead_rowmajor(_c=None):
        st.spec_lm_head_stats(lm_x, lm_w, T, outputs=lm_out, workspace=lm_ws, status=lm_st)

    for _ in range(3):
        lmhead()
    torch.cuda.synchronize()
    assert int(lm_st.item()) == 0
    g_p, g_c = capture(paged, pcs), capture(compact, bufs)
    g_f, g_v = capture(filtered, bufs), capture(plain, bufs)
    g_tb, g_tx = capture(build, tcs), capture(expand_all, tcs)
    # temperature-0 verification straight from the fused head's argmax (no logit row anywhere)
    g_st = torch.zeros((B,), dtype=torch.int32, device=dev)
    g_out = st.spec_tree_verify_greedy(lm_out["argmax"].view(B, N), bufs[0]["tokens"],
                                       bufs[0]["parent"], V, status=g_st)

    def lm_greedy(_c=None):
        lmhead()
        st.spec_tree_verify_greedy(lm_out["argmax"].view(B, N), bufs[0]["tokens"],
                                   bufs[0]["parent"], V, outputs=g_out, status=g_st)

    lm_greedy()
    torch.cuda.synchronize()
    assert int(g_st.sum()) == 0
    # verification from the LM head's statistics at this workload's shape (hidden size Hq D):
    # lattice operands (exact logits) with an EAGLE-style draft, so that the walk accepts and
    # rejects as it would on the plain path; the head (> 2 x L2) is read from HBM every pass
    hcase = W.make_head_verify_case(cfg, lm_h, T, seed=args.seed + 5)
    h_dev = {"h": to_dev(hcase.hidden).view(torch.bfloat16),
             "w": to_dev(hcase.head).view(torch.bfloat16), "p": to_dev(hcase.draft_probs),
             "t": to_dev(hcase.tree_tokens), "par": to_dev(hcase.tree_parent),
             "u": to_dev(hcase.uniforms)}
    h_dev["wp"] = st.spec_lm_head_pack(h_dev["w"])
    h_ws = torch.empty((st.spec_tree_verify_head_workspace(B, N, lm_h, V, hcase.max_depth),),
                       dtype=torch.uint8, device=dev)
    h_st = torch.zeros((B,), dtype=torch.int32, device=dev)
    h_out = st.spec_tree_verify_head(h_dev["h"], h_dev["wp"], h_dev["p"], h_dev["t"],
                                     h_dev["par"], h_dev["u"], T, hcase.max_depth,
                                     packed_vocab=V, workspace=h_ws, status=h_st)

    def head_verify(_c=None):
        st.spec_tree_verify_head(h_dev["h"], h_dev["wp"], h_dev["p"], h_dev["t"], h_dev["par"],
                                 h_dev["u"], T, hcase.max_depth, packed_vocab=V, outputs=h_out,
                                 workspace=h_ws, status=h_st)

    torch.cuda.synchronize()
    assert int(h_st.sum()) == 0
    reps_lm = 20
    g_hv = capture(head_verify, [None] * 5)
    g_lm = capture(lmhead, [None] * reps_lm)
    g_lr = capture(lmhead_rowmajor, [None] * reps_lm)
    g_lg = capture(lm_greedy, [None] * reps_lm)
    g_gr = capture(lambda _c: st.spec_tree_verify_greedy(
        lm_out["argmax"].view(B, N), bufs[0]["tokens"], bufs[0]["parent"], V, outputs=g_out,
        status=g_st), [None] * reps_lm)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g_p.replay()
        g_c.replay()
        g_f.replay()
        g_v.replay()
        g_tb.replay()
        g_tx.replay()
        g_lm.replay()
        g_lr.replay()
        g_lg.replay()
        g_gr.replay()
        g_hv.replay()
    torch.cuda.synchronize()
    reps = max(1, 600 // ncp)
    p_ms = timed(lambda: [g_p.replay() for _ in range(reps)]) / (reps * ncp)
    reps_f = max(1, 600 // len(bufs))
    f_ms = timed(lambda: [g_f.replay() for _ in range(reps_f)]) / (reps_f * len(bufs))
    v_ms = timed(lambda: [g_v.replay() for _ in range(reps_f)]) / (reps_f * len(bufs))
    filt_bytes = 2 * B * N * V * 4  # the logits read once, the filtered logits written once
    reps_t = max(1, 300 // ncp_t)
    tb_ms = timed(lambda: [g_tb.replay() for _ in range(reps_t)]) / (reps_t * ncp_t)
    tx_ms = timed(lambda: [g_tx.replay() for _ in range(reps_t)]) / (reps_t * ncp_t)
    tree_bytes = tcase.draft_rows.nbytes  # every draft row read once
    lm_ms = timed(lambda: [g_lm.replay() for _ in range(10)]) / (10 * reps_lm)
    lr_ms = timed(lambda: [g_lr.replay() for _ in range(10)]) / (10 * reps_lm)
    lg_ms = timed(lambda: [g_lg.replay() for _ in range(10)]) / (10 * reps_lm)
    gr_ms = timed(lambda: [g_gr.replay() for _ in range(10)]) / (10 * reps_lm)
    hv_ms = timed(lambda: [g_hv.replay() for _ in range(10)]) / (10 * 5)
    # row passes that processed a node: per sequence, the walk's nodes where it did not move on to
    # the first child (a rejected first child, or the terminal node)
    h_len = h_out["accept_len"].cpu().numpy()
    h_nodes = h_out["accepted_nodes"].cpu().numpy()
    passes = []
    for b in range(B):
        par_b = hcase.tree_parent[b]
        walk = [0] + [int(x) for x in h_nodes[b, :max(int(h_len[b]), 0)]]
        stops = 1
        for c, nxt in zip(walk[:-1], walk[1:]):
            first = next(k for k in range(c + 1, N) if par_b[k] == c)
            stops += 0 if nxt == first else 1
        passes.append(stops)
    head_bytes = V * lm_h * 2
    internal = int(sum(len(set(int(x) for x in hcase.tree_parent[b, 1:])) for b in range(B)))
    lm_bytes = lm_w.numel() * 2 + lm_x.numel() * 2 + lm_m * 12  # head, hidden, statistics
    lm_flops = 2.0 * lm_m * lm_h * V
    fil_gbs = filt_bytes / ((f_ms - v_ms) * 1e-3) / 1e9 if f_ms > v_ms else None
    reps_c = max(1, 600 // len(bufs))
    c_ms = timed(lambda: [g_c.replay() for _ in range(reps_c)]) / (reps_c * len(bufs))
    _, Hkv, _, D = bufs[0]["k"].shape
    lens = bufs[0]["vout"]["accept_len"].cpu().numpy()
    moved = int(np.maximum(lens, 0).sum()) * Hkv * D * 2 * 2 * 2  # K and V rows, read + write
    p_gbs = attn_bytes / (p_ms * 1e-3) / 1e9
    return {
        "paged_attention": {"page_size": page, "us_per_call": p_ms * 1e3, "achieved_gbs": p_gbs,
                            "frac": p_gbs / hbm_gbs, "contiguous_us_per_call": attn_ms * 1e3,
                            "algorithmic_bytes": attn_bytes, "copies": ncp,
                            "kernel": "tree_attn_kernel, boxes addressed through the block table"},
        "kv_compact": {"us_per_call": c_ms * 1e3, "accept_len": lens.tolist(),
                       "algorithmic_bytes": moved,
                       "achieved_gbs": moved / (c_ms * 1e-3) / 1e9,
                       "note": "latency-bound: a few KB to a few hundred KB per call"},
        "filtered_verify": {"top_k": top_k, "top_p": top_p, "temperature": T,
                            "us_per_call": f_ms * 1e3, "plain_verify_us_per_call": v_ms * 1e3,
                            "filter_us_per_call": (f_ms - v_ms) * 1e3,
                            "filter_algorithmic_bytes": filt_bytes, "filter_achieved_gbs": fil_gbs,
                            "filter_frac": fil_gbs / hbm_gbs if fil_gbs else None,
                            "kernel": "filter_kernel (cluster per row, row in shared memory)",
                            "note": "filter kernel time = filtered call - plain call (same "
                                    "copies, same temperature); latency-bound"},
        "tree_build": {"K": tK, "depth": tD, "nodes": N, "rows_per_sequence": 1 + (tD - 1) * tK,
                       "us_per_tree": tb_ms * 1e3, "expand_us_all_levels": tx_ms * 1e3,
                       "finalize_us": (tb_ms - tx_ms) * 1e3, "algorithmic_bytes": tree_bytes,
                       "achieved_gbs": tree_bytes / (tx_ms * 1e-3) / 1e9,
                       "frac": tree_bytes / (tx_ms * 1e-3) / 1e9 / hbm_gbs, "copies": ncp_t,
                       "kernel": "expand_kernel (one CTA per draft row, six launches), "
                                 "finalize_kernel",
                       "note": "expand rate = draft-row bytes / time of the six expand launches"},
        "lm_head": {"rows": lm_m, "hidden": lm_h, "vocab": V, "us_per_call": lm_ms * 1e3,
                    "algorithmic_bytes": lm_bytes,
                    "achieved_gbs": lm_bytes / (lm_ms * 1e-3) / 1e9,
                    "frac": lm_bytes / (lm_ms * 1e-3) / 1e9 / hbm_gbs,
                    "tflops": lm_flops / (lm_ms * 1e-3) / 1e12,
                    "tensor_frac": lm_flops / (lm_ms * 1e-3) / 1e12 / tc_tflops,
                    "rowmajor_us_per_call": lr_ms * 1e3,
                    "greedy_verify_pipeline_us": lg_ms * 1e3,
                    "greedy_verify_us": gr_ms * 1e3,
                    "kernel": "lm_head_kernel (tcgen05, 128 x 256 tiles, tile-major head) + "
                              "lm_head_combine_kernel; pipeline: + verify_greedy_kernel (T = 0 "
                              "verification of the workload's tree from the argmax)",
                    "note": "weights generated on the device (seeded), bf16; the logit matrix is "
                            "never written"},
        "verify_head": {"hidden": lm_h, "vocab": V, "temperature": T,
                        "max_depth": hcase.max_depth, "us_per_call": hv_ms * 1e3,
                        "row_passes_used": passes, "row_passes_launched": hcase.max_depth + 1,
                        "mean_accept_len": float(np.mean(h_len)),
                        "head_bytes_read": head_bytes * (1 + max(passes)),
                        "logit_row_bytes": 4 * V * int(sum(passes)),
                        "logit_row_bytes_plain_verify": 4 * V * internal,
                        "logit_matrix_bytes_not_written": 4 * V * B * N,
                        "lm_head_stats_us": lm_ms * 1e3,
                        "kernel": "head_prep_kernel, lm_head_kernel + lm_head_combine_kernel "
                                  "(statistics of every node), head_walk_kernel, then per row "
                                  "pass lm_head_kernel (rows of the pending nodes) and "
                                  "verify_head_step_kernel (which continues the walk); "
                                  "head_finish_kernel",
                        "note": "lattice hidden states and head (exact logits), EAGLE-style "
                                "draft; one row pass = one more read of the head"},
        "peak_gbs": hbm_gbs,
    }


# ------------------------------------------------------------------------------------------------
# the other workloads: batched GQA, long context, the stress sweep, temperature 0
# ------------------------------------------------------------------------------------------------
# (key, configuration, temperature, batch override or None, timed: attention + verification step)
OTHER_WORKLOADS = (
    ("eagle_vicuna7b_T0", "eagle_vicuna7b", 0.0, None, True),
    ("llama3_8b_gqa", "llama3_8b_gqa", 0.7, None, True),
    ("llama70b_longctx", "llama70b_longctx", 1.0, None, True),
    ("stress_T1", "stress", 1.0, None, True),
    ("stress_T0", "stress", 0.0, 16, False),
    ("stress_T0.5", "stress", 0.5, 16, False),
    ("stress_T1.5", "stress", 1.5, 16, False),
)


def cpu_leg_workload(spec):
    """CPU-baseline leg of one of the other workloads (a spawned worker process, one thread):
    draws the workload's verification inputs and times the fp64 oracle verifying every sequence of
    them.  Returns the inputs (for the GPU side), the oracle's outputs (for the near-tie count and
    the agreement check) and the oracle's time."""
    name, T, seed, batch = spec
    from oracle import verify as OV
    from speculative_decoding_token_spec_gb300 import workloads as W
    cfg = W.config(name) if batch is None else W.config(name, B=batch)
    vc = W.make_verify_case(cfg, T, seed=seed)
    t0 = time.perf_counter()
    ref = OV.tree_verify(vc.target_logits, vc.draft_probs, vc.tree_tokens, vc.tree_parent,
                         vc.uniforms, T)
    dt = time.perf_counter() - t0
    keep = ("accept_len", "accepted_tokens", "bonus", "near_tie", "status")
    return {"case": vc, "oracle": {k: ref[k] for k in keep}, "oracle_s": dt}


def start_cpu_legs(seed):
    """Starts the other workloads' CPU legs in a spawned pool (no fork after CUDA is up)."""
    import concurrent.futures
    import multiprocessing
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 4
    env1 = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}
    old = {k: os.environ.get(k) for k in env1}
    os.environ.update(env1)  # inherited by the spawned workers
    try:
        pool = concurrent.futures.ProcessPoolExecutor(
            max_workers=max(1, min(len(OTHER_WORKLOADS), cores - 2)),
            mp_context=multiprocessing.get_context("spawn"))
        futs = {key: pool.submit(cpu_leg_workload, (name, T, seed, batch))
                for key, name, T, batch, _ in OTHER_WORKLOADS}
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return pool, futs


def acceptance_stats(accept_len, N_depth):
    """Mean accepted length, emitted tokens per step and the acceptance rate at each depth d
    (sequences that accepted a depth-d node / sequences whose walk reached depth d - 1)."""
    import numpy as np
    a = np.asarray(accept_len)
    a = a[a >= 0]
    per_depth = []
    for d in range(1, N_depth + 1):
        reached = int((a >= d - 1).sum())
        per_depth.append(round(float((a >= d).sum()) / reached, 4) if reached else None)
    return {"mean_accept_len": float(a.mean()) if len(a) else None,
            "tokens_per_step": float(a.mean() + 1) if len(a) else None,
            "accept_rate_per_depth": per_depth, "sequences": int(len(a))}


def measure_other_workloads(args, dev, futs, hbm_gbs, tc_tflops, timed, L2):
    """Per workload: attention, verification and step times from CUDA graphs (inputs larger than
    L2, or rotated over copies that are), the algorithmic bytes and HBM (or tensor) fractions, the
    verification statistics of the GPU outputs, and the oracle leg's near-tie count, agreement and
    time."""
    import numpy as np
    import torch
    import speculative_decoding_token_spec_gb300 as st
    from speculative_decoding_token_spec_gb300 import workloads as W
    out = {}
    s = torch.cuda.Stream(device=dev)
    for key, name, T, batch, timed_step in OTHER_WORKLOADS:
        leg = futs[key].result()
        vc = leg["case"]
        cfg = W.config(name) if batch is None else W.config(name, B=batch)
        B, N, V = vc.target_logits.shape
        lens, par, Lmax = W.attention_layout(cfg, args.seed)
        assert np.array_equal(par, vc.tree_parent)
        Hq, Hkv, D = cfg.Hq, cfg.Hkv, cfg.D
        to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        ver_bytes_per_copy = vc.target_logits.nbytes + (vc.draft_probs.nbytes if T > 0 else 0)
        kv_bytes = 2 * B * Hkv * Lmax * D * 2 if timed_step else 0
        per_copy = ver_bytes_per_copy + kv_bytes
        copies = max(1, min(9, math.ceil(2 * L2 / per_copy)))
        gen = torch.Generator(device=dev)
        gen.manual_seed(1000 + args.seed)
        bufs = []
        for _ in range(copies):
            c = {"logits": to_dev(vc.target_logits), "probs": to_dev(vc.draft_probs) if T > 0 else None,
                 "tokens": to_dev(vc.tree_tokens), "parent": to_dev(vc.tree_parent),
                 "unif": to_dev(vc.uniforms), "st_v": torch.zeros((B,), dtype=torch.int32, device=dev)}
            c["ws_v"] = torch.empty((max(st.spec_tree_verify_workspace(B, N, V), 16),),
                                    dtype=torch.uint8, device=dev)
            i32 = dict(dtype=torch.int32, device=dev)
            c["vout"] = {"accept_len": torch.empty((B,), **i32),
                         "accepted_tokens": torch.empty((B, N), **i32),
                         "bonus": torch.empty((B,), **i32),
                         "accepted_nodes": torch.empty((B, N), **i32)}
            if timed_step:
                rnd = lambda *shape: torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)  # noqa: E731,E501
                c["q"], c["k"], c["v"] = rnd(B, N, Hq, D), rnd(B, Hkv, Lmax, D), rnd(B, Hkv, Lmax, D)
                c["lens"] = to_dev(lens)
                c["out"] = torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev)
                c["lse"] = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
                c["st_a"] = torch.zeros((B,), dtype=torch.int32, device=dev)
            bufs.append(c)

        def attn(c):
            st.spec_tree_attention(c["q"], c["k"], c["v"], c["lens"], c["parent"],
                                   softmax_scale=1.0 / math.sqrt(D), out=c["out"], out_lse=c["lse"],
                                   status=c["st_a"])

        def verify(c):
            st.spec_tree_verify(c["logits"], c["probs"], c["tokens"], c["parent"], c["unif"], T,
                                outputs=c["vout"], workspace=c["ws_v"], status=c["st_v"])

        def step(c):
            attn(c)
            verify(c)

        fns = {"verify": verify}
        if timed_step:
            fns.update({"attn": attn, "step": step})
        for _ in range(3):
            for c in bufs:
                for f in fns.values():
                    f(c)
        torch.cuda.synchronize()
        reps_per_graph = max(1, -(-12 // copies))
        graphs = {}
        s.wait_stream(torch.cuda.current_stream())
        for k, f in fns.items():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for _ in range(reps_per_graph):
                        for c in bufs:
                            f(c)
            graphs[k] = g
        torch.cuda.current_stream().wait_stream(s)
        for g in graphs.values():
            g.replay()
            g.replay()
        torch.cuda.synchronize()
        calls = reps_per_graph * copies
        us = {}
        replays = 20  # a few hundred calls per timed region
        for k, g in graphs.items():
            us[k] = timed(lambda: [g.replay() for _ in range(replays)]) * 1e3 / (replays * calls)
        o = {k: v.cpu().numpy() for k, v in bufs[0]["vout"].items()}
        o["status"] = bufs[0]["st_v"].cpu().numpy()
        ref = leg["oracle"]
        near = ref["near_tie"]
        agree = sum(1 for b in range(B) if not near[b]
                    and o["accept_len"][b] == ref["accept_len"][b]
                    and o["bonus"][b] == ref["bonus"][b]
                    and np.array_equal(o["accepted_tokens"][b], ref["accepted_tokens"][b]))
        internal = sum(len(np.unique(par[b, 1:])) for b in range(B)) if N > 1 else 0
        ver_bytes = internal * 4 * V * (2 if T > 0 else 1) + B * 4 * V * (2 if T > 0 else 1)
        path_form = B * N * V * 4 > (64 << 20)
        read_bytes = None
        if path_form:
            read_bytes = 0
            for b in range(B):
                for j in [0] + [int(x) for x in o["accepted_nodes"][b, :max(int(o["accept_len"][b]), 0)]]:
                    kids = bool((par[b, 1:] == j).any())
                    read_bytes += 4 * V * (2 if (T > 0 and kids) else 1)
        depth = int(max(W.config(name).depth, 1))
        e = {"workload": workload_name(cfg, T), "temperature": T,
             "verify_us": us["verify"],
             "verify_form": "path only (one cluster per sequence)" if path_form
                            else "every node at once",
             "verify_algorithmic_bytes": ver_bytes, "verify_read_bytes": read_bytes,
             "verify_read_gbs": read_bytes / (us["verify"] * 1e-6) / 1e9 if read_bytes else None,
             "verification": acceptance_stats(o["accept_len"], depth),
             "status_nonzero": int((o["status"] != 0).sum()),
             "cpu_baseline": {"kind": "oracle", "cores": 1,
                              "value": B / leg["oracle_s"], "unit": "sequences/s (verification)",
                              "sample": f"fp64 oracle verification of all {B} sequences",
                              "near_ties": int(near.sum()), "compared": int((~near).sum()),
                              "gpu_agrees": int(agree)},
             "copies": copies, "calls_per_region": calls * replays}
        if timed_step:
            kv = sum(Hkv * (int(L) + N) * D * 2 * 2 for L in lens)
            attn_bytes = kv + 2 * B * N * Hq * D * 2 + B * Hq * N * 4
            flops = sum(4 * Hq * N * (int(L) + N) * D for L in lens)
            step_s = us["step"] * 1e-6
            e.update({"nodes_per_s": B * N / step_s, "step_us": us["step"], "attn_us": us["attn"],
                      "attn_algorithmic_bytes": attn_bytes,
                      "attn_gbs": attn_bytes / (us["attn"] * 1e-6) / 1e9,
                      "attn_frac": attn_bytes / (us["attn"] * 1e-6) / 1e9 / hbm_gbs,
                      "attn_tflops": flops / (us["attn"] * 1e-6) / 1e12,
                      "attn_tensor_frac": flops / (us["attn"] * 1e-6) / 1e12 / tc_tflops,
                      # the bytes the step reads: the path form reads only the walk's rows
                      "step_hbm_frac": (attn_bytes + (read_bytes if path_form else ver_bytes))
                                       / (hbm_gbs * 1e9) / step_s,
                      "step_hbm_frac_all_rows": (attn_bytes + ver_bytes) / (hbm_gbs * 1e9)
                                                / step_s,
                      "dominant_kernel": "tree_attn_kernel" if us["attn"] >= us["verify"]
                                         else "verify_kernel"})
        out[key] = e
        del bufs, graphs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out["note"] = ("per-call times from CUDA graphs of back-to-back calls (inputs larger than 2 x L2 "
                   "or rotated over copies that are); verify_algorithmic_bytes counts every "
                   "internal node's rows (the all-nodes count), verify_read_bytes the rows the path "
                   "form actually reads; step_hbm_frac counts the bytes the step reads (the path "
                   "form's rows), step_hbm_frac_all_rows every internal row (above 1 where the "
                   "path form skips rows); Q/K/V drawn on the device (seeded), the verification "
                   "inputs by the workload generator; cpu_baseline: the fp64 oracle's "
                   "verification of the same inputs (near ties counted, the GPU's tokens compared "
                   "outside them)")
    return out



def profiled_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    src = os.path.join(ROOT, "speculative_decoding_token_spec_gb300", "csrc", "tree_attention.cu")
    try:
        kv = {}
        with open(path) as f:
            for l in f:
                if ":" in l:
                    k, v = l.split(":", 1)
                    kv[k.strip()] = v.strip()
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if kv.get("source_sha256") != sha:
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------------------------------------
# reference arm: the CPU oracle on the same metric
# ------------------------------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    budget = min(60.0, max(10.0, 0.02 * (args.steps + args.warmup)))
    r = run_cpu_oracle(args.config, args.temperature, args.seed, steps=args.steps, budget=budget)
    from speculative_decoding_token_spec_gb300 import workloads as W
    cfg = W.config(args.config)
    line = {
        "impl": "reference", "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["seconds"] * 1e3 / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the EAGLE static-tree workload, no datasets)",
        "config": {"workload": workload_name(cfg, args.temperature),
                   "parallelism": "cpu oracle, rank 0 only"},
        "cpu_baseline": {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"], "cpu": cpu_model()},
        "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


def main():
    args = parse_args()
    if args.cpu_child:
        cpu_oracle_child(args.cpu_child)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
