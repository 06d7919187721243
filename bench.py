"""Benchmark: one tree-verification pass per step.  The default workload is
batched serving (B=64, 32/8 heads, D=128, bf16, 16-token pages with a random
block table, prefixes U[256, 16384], trees of U[8, 64] nodes, V=32000, greedy
verification, then KV commit), the largest single-GPU configuration and the
one whose attention is bound by HBM.

A step = spec_tree_mask_build + spec_tree_attention + spec_tree_verify_{greedy,
stochastic} + spec_kv_commit over one batch whose inputs are already in HBM
(the tree K/V resident in their slots).  Inputs larger than L2 (one 2.2 GB
set for batched serving; three rotating ~205 MB sets for the decode layer and
the ensemble) make every step read from DRAM.  The e2e figure adds, every
step, the host-to-device copy of the step's inputs including the tree K/V
rows, their spec_kv_append, and the read-back of the emitted tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload 1|2|3|4]

Prints one JSON line.  Metric: tree-verify tokens/s = tokens emitted by the
verifier per second of pass time.  For N > 1 (torchrun) every rank runs an
independent replica (requests are independent; no collective on the data path).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify tokens/s"
UNIT = "tokens/s"
# --workload: 3 (batched serving) is the default line; the others give the same
# contract line for the decode layer, the wide-ensemble tree and one
# linear-vs-tree sweep point
WORKLOADS = {
    1: dict(desc="Llama-style decode layer: B=8, 32 query / 8 KV heads, head_dim 128, bf16, prefix 2048, 64-node "
                 "expansion trees (4,2,2,1,1,1,1,1) per request, V=32000, stochastic verification, KV commit",
            mode="stochastic", sets=3),
    2: dict(desc="wide ensemble tree: B=1, 64 query / 8 KV heads, head_dim 128, bf16, prefix 8192, 256-node merge "
                 "of 4 random depth-8 trees, V=128256, stochastic verification, KV commit",
            mode="stochastic", sets=3),
    3: dict(desc="batched serving: B=64, 32 query / 8 KV heads, head_dim 128, bf16, 16-token pages, random block "
                 "table, prefix U[256,16384], trees U[8,64] nodes, V=32000, greedy verification, KV commit",
            mode="greedy", sets=1),
    4: dict(desc="linear-vs-tree sweep point: chains of K+1=9 nodes, B=64, 32 query / 8 KV heads, head_dim 128, bf16, "
                 "prefix 4096, V=32000, draft = 0.7 p + 0.3 r, stochastic verification, KV commit",
            mode="stochastic", sets=1),
}


def make_workload(which, seed_base, i):
    import workloads as W
    if which == 1:
        return W.config1(seed=1001 + seed_base + i)
    if which == 2:
        return W.config2(seed=1002 + seed_base + i)
    if which == 3:
        return W.config3(seed=1003 + seed_base + i)
    return W.config4(K=8, B=64, tree="chain", alpha=0.3, seed=1004 + seed_base + i)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(w, stats, mode="stochastic"):
    """Per-launch algorithmic bytes of each kernel (formulas of the design)."""
    s = 2 if w.dtype == 1 else 4
    Wd = (w.n_max + 63) // 64
    n = (w.tree_off[1:] - w.tree_off[:-1]).tolist()
    P = w.prefix_len.tolist()
    attn = sum(2 * w.Hkv * w.D * s * (P[b] + n[b]) + 2 * n[b] * w.Hq * w.D * s + 8 * n[b] * Wd for b in range(w.B))
    # the walk reads the target row of every node it reaches, and the draft row
    # of every reached node where a child was rejected
    verify = 4 * w.V * (stats["walk_rows"] + (stats["rejecting_nodes"] if mode == "stochastic" else 0))
    mask = 4 * w.T + 12 * w.T + 8 * w.T * Wd
    commit = 2 * 2 * w.Hkv * w.D * s * stats["moved_rows"]
    # the tree's K and V rows: read from the caller's arrays, written to their slots
    append = 2 * 2 * w.T * w.Hkv * w.D * s
    return dict(mask=mask, attention=attn, verify=verify, commit=commit, append=append)


def attention_flops(w):
    """4 * D * Hq * sum over nodes u of (P_b + depth(u) + 1): every unmasked key."""
    par = w.parent.tolist()
    off = w.tree_off.tolist()
    total = 0
    for b in range(w.B):
        depth = {}
        for i in range(off[b + 1] - off[b]):
            p = par[off[b] + i]
            depth[i] = 0 if p < 0 else depth[p] + 1
            total += int(w.prefix_len[b]) + depth[i] + 1
    return 4 * w.D * w.Hq * total


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def _tree_stats(w, accept_paths):
    """Rows the verifier's walk reads and rows the commit moves, from the
    accepted paths: every path node's target row; the draft row of a path node
    whose accepted child is not its first child, or of the last path node when
    it has children (all of them rejected)."""
    par = w.parent.tolist()
    off = w.tree_off.tolist()
    walk_rows = rejecting = moved = 0
    for b, row in enumerate(accept_paths):
        n = off[b + 1] - off[b]
        kids = [[] for _ in range(n)]
        for c in range(1, n):
            kids[par[off[b] + c]].append(c)
        path = [p for p in row if p >= 0]
        walk_rows += len(path)
        for i, u in enumerate(path):
            nxt = path[i + 1] if i + 1 < len(path) else None
            if kids[u] and (nxt is None or kids[u][0] != nxt):
                rejecting += 1
        moved += sum(1 for i, p in enumerate(row) if p >= 0 and p != i)
    return dict(walk_rows=walk_rows, rejecting_nodes=rejecting, moved_rows=moved)


class ClockSampler:
    """SM clock and clock-event reasons of one GPU, sampled every ~2 ms in a
    background thread through NVML (read-only queries), with nvidia-smi as a
    fallback when NVML cannot be loaded."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        import threading
        self.dev = device_index
        self.samples = []
        self.stop = threading.Event()
        self.thread = None
        self.proc = None

    def _nvml(self):
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        assert nv.nvmlInit_v2() == 0
        h = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            assert nv.nvmlDeviceGetHandleByIndex_v2(self.dev, ctypes.byref(h)) == 0
        return nv, h

    def _run(self):
        import ctypes
        nv, h = self.nv, self.h
        mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            ok = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0  # NVML_CLOCK_SM
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            get_reasons(h, ctypes.byref(rs))
            if ok:
                self.samples.append((float(mhz.value), float(mx.value), int(rs.value)))
            time.sleep(0.002)

    def __enter__(self):
        import threading
        try:
            self.nv, self.h = self._nvml()
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except Exception:
            self.thread = None
            try:
                q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                     "clocks_event_reasons.sw_power_cap")
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "100"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None
        return self

    def __exit__(self, *a):
        self.stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = [0x8, 0x40, 0x20, 0x4]
            for l in out.splitlines():
                f = [x.strip() for x in l.split(",")]
                try:
                    r = sum(bit for bit, v in zip(names, f[2:6]) if v.lower().startswith("active"))
                    self.samples.append((float(f[0]), float(f[1]), r))
                except (ValueError, IndexError):
                    continue

    def mark_timed_end(self):
        """Record where the timed region's samples end (the sampler keeps going)."""
        self.timed_n = len(self.samples)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({name for _, _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        out = {"sm_mhz": statistics.median(x[0] for x in self.samples),
               "sm_max_mhz": max(x[1] for x in self.samples), "reasons": reasons, "samples": len(self.samples),
               "source": "nvml" if self.thread is not None else "nvidia-smi"}
        tn = getattr(self, "timed_n", None)
        if tn is not None:
            timed = self.samples[:tn]
            out["window"] = ("the timed region and the kernel-timing replays right after it (same kernels, same "
                             "inputs)")
            out["timed_region_samples"] = len(timed)
            out["timed_region_sm_mhz"] = statistics.median(x[0] for x in timed) if timed else None
        return out


def _oracle_request(item):
    """One request's full pass in the oracle (runs in a spawned worker)."""
    import time as _time
    import numpy as np
    import oracle as O
    (par, toff, n_max, q, kc, vc, bt, bs, prefix, Hq, Hkv, D, dtype, scale, mode, logits, draft, tokens, uni) = item
    t0 = _time.perf_counter()
    O.mask_build(par, toff, n_max)
    O.tree_attention(q, kc, vc, bt, bs, prefix, toff, par, n_max, Hq, Hkv, D, dtype, scale)
    if mode == "greedy":
        r = O.verify_greedy(logits, tokens, par, toff, n_max)
    else:
        r = O.verify_stochastic(logits, draft, tokens, par, toff, uni, n_max)
    O.kv_commit(kc, vc, bt, bs, prefix, r["path"], r["accept_len"], Hkv, D, dtype, np.zeros(1, np.int32))
    return int(r["n_emitted"][0]), _time.perf_counter() - t0


def _oracle_items(w, mode, count):
    """Per-request oracle inputs of requests 0 .. count-1, each with a
    one-request cache made of the pages it owns."""
    import numpy as np
    import torch

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    items = []
    for b in range(count):
        lo, hi = int(w.tree_off[b]), int(w.tree_off[b + 1])
        nblk = int((w.prefix_len[b] + (hi - lo) + w.block_size - 1) // w.block_size)
        pages = w.block_table[b, :nblk].long()
        kc, vc = bits(w.k_cache[pages]), bits(w.v_cache[pages])
        items.append((w.parent[lo:hi].numpy(), np.array([0, hi - lo], np.int32), w.n_max, bits(w.q[lo:hi]), kc, vc,
                      np.arange(nblk, dtype=np.int32)[None, :], w.block_size, w.prefix_len[b:b + 1].numpy(), w.Hq,
                      w.Hkv, w.D, w.dtype, w.scale, mode, w.p_logits[lo:hi].numpy(),
                      None if mode == "greedy" else w.q_probs[lo:hi].numpy(), w.tokens[lo:hi].numpy(),
                      None if mode == "greedy" else w.uniforms[lo:hi].numpy().view(np.uint32)))
    return items


def cpu_workers(w):
    """Host processes for the oracle baseline: one per request, up to the
    host's cores and 8."""
    return max(1, min(w.B, os.cpu_count() or 1, 8))


def run_cpu_baseline(w, mode="stochastic", workers=1, pool=None):
    """The oracle as it stands (plain C, one thread per process) on a bounded
    sample of the same workload: the full pass (mask, attention, verify in
    `mode`, commit) of requests 0 .. workers-1, one spawned process per
    request.  Returns (tokens/s, sample description, seconds, processes)."""
    items = _oracle_items(w, mode, workers)
    t0 = time.perf_counter()
    res = pool.map(_oracle_request, items) if pool is not None else [_oracle_request(it) for it in items]
    dt = time.perf_counter() - t0
    tokens = sum(r[0] for r in res)
    what = (f"requests 0..{workers - 1} of the batch ({workers} of {w.B}), one host process each, full pass in the "
            f"oracle, {dt:.2f} s wall")
    return tokens / dt, what, dt, workers


def oracle_pool(workers):
    """A spawned pool (never forked: the parent has a CUDA context), warmed up
    so that the timed map excludes process start-up."""
    if workers <= 1:
        return None
    import multiprocessing as mp
    pool = mp.get_context("spawn").Pool(workers)
    pool.map(_warm, range(workers))
    return pool


def _warm(_):
    import oracle as O
    O.lib()
    return 0


def bench_reference(args):
    """--impl reference: the CPU oracle as the reference arm (timed on the host)."""
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    w = make_workload(args.workload, args.seed, 0)
    workers = cpu_workers(w)
    pool = oracle_pool(workers)
    times, toks = [], 0.0
    for i in range(args.warmup + args.steps):
        v, sample, dt, _ = run_cpu_baseline(w, args.mode, workers, pool)
        if i >= args.warmup:
            times.append(dt)
            toks += v * dt
    if pool is not None:
        pool.close()
        pool.join()
    total = sum(times)
    value = toks / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32", "data": "synthetic",
            "config": {"workload": wl["desc"], "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def aggregate_replicas(elapsed_ms, tokens, device):
    """Whole-job figures of independent replicas: the slowest rank's time and
    the tokens of all ranks (no collective touches the data path)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return elapsed_ms, tokens
    t = torch.tensor([elapsed_ms, tokens], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[1])


def bench_gpu(args):
    import torch
    import workloads as W
    import tree_speculative_verification_spec_gb300 as S
    from tree_speculative_verification_spec_gb300 import build as B_
    from tree_speculative_verification_spec_gb300.pipeline import DeviceBatch, VerifyPass

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    B_.build()
    S.lib()
    dev = torch.device("cuda", local)

    wl = WORKLOADS[args.workload]
    n_sets = wl["sets"]
    sets, passes, works = [], [], []
    for i in range(n_sets):
        w = make_workload(args.workload, args.seed + 97 * rank, i)
        works.append(w)
        d = DeviceBatch.from_workload(w, device=dev)
        sets.append(d)
        vp = VerifyPass(d)
        if args.temperature is not None:
            vp.inv_temp = torch.full((w.B,), 1.0 / args.temperature, dtype=torch.float32, device=dev)
        vp.q_layout = S.SPEC_Q_PER_CHILD if args.q_per_child else S.SPEC_Q_PER_PARENT
        passes.append(vp)
    torch.cuda.synchronize()

    stages = ("mask", "attention", "verify", "commit")

    def step(vp, skip=None):
        """One pass (optionally without one stage, for the differential timing)."""
        for name, fn in (("mask", vp.mask_build), ("attention", lambda: vp.attention(args.attn_flags)),
                         ("verify", lambda: vp.verify(args.mode)), ("commit", vp.commit)):
            if name != skip:
                fn()

    # eager warm-up (first calls set kernel attributes and look up driver entry points)
    for i in range(args.warmup):
        step(passes[i % n_sets])
    torch.cuda.synchronize()

    def capture(skip=None):
        """One CUDA graph of one pass per input set (no event nodes inside)."""
        cap = torch.cuda.Stream(dev)
        gs = []
        for i in range(n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step(passes[i], skip)
            gs.append(g)
        torch.cuda.synchronize()
        return gs

    stream = torch.cuda.current_stream(dev)

    def timed(graphs):
        """K replays bracketed by CUDA events on the replay stream (barrier and
        synchronize on both sides); returns milliseconds."""
        for i in range(args.warmup):
            graphs[i % n_sets].replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(args.steps):
            graphs[i % n_sets].replay()
        b.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return a.elapsed_time(b)

    graphs = capture()
    # The clock sampler runs through the timed region and the kernel-timing
    # legs right after it (hundreds of replays of the same kernels), so that
    # the clock record spans more than the K timed steps.
    with ClockSampler(local) as clk:
        elapsed_ms = timed(graphs)
        clk.mark_timed_end()
        # per-kernel launch durations: the same K steps without that kernel,
        # timed the same way right after; duration = (full - without) / K
        stage = {}
        for k in stages:
            stage[k] = max(0.0, (elapsed_ms - timed(capture(skip=k))) / args.steps)
        # each kernel alone: one graph per stage of input set 0, replayed with
        # an L2 flush (a write of twice the L2 size) before every replay, each
        # replay bracketed by its own CUDA events
        tree_kv = [t.to(dev) for t in W.tree_kv_rows(works[0], 11)]
        iso = isolated_times(passes[0], args, dev, stream, tree_kv)
    dom = max(("attention", "verify"), key=lambda k: stage[k])

    # emitted tokens per step (verify inputs do not change between steps of one set)
    tokens_per_set = [int(p.n_emitted[:p.batch.B].sum()) for p in passes]
    status_ok = all(int(p.status[:p.batch.B].abs().sum()) == 0 for p in passes)
    tokens = sum(tokens_per_set[i % n_sets] for i in range(args.steps))
    elapsed_ms, tokens = aggregate_replicas(elapsed_ms, float(tokens), dev)
    value = tokens / (elapsed_ms / 1e3)

    # --- e2e through the C ABI with host buffers: per step, H2D of the step's
    # inputs from pinned memory, the five calls, D2H of the emitted tokens; the KV
    # cache is resident state.
    e2e = run_e2e(args, works, sets, passes, stream, dev, n_sets)

    # --- roofline of the dominant kernel
    peak, peak_kind = _peaks()
    w0 = works[0]
    stats = _tree_stats(w0, passes[0].path[:w0.B].tolist())
    algo = algorithmic_bytes(w0, stats, args.mode)
    avg = stage
    kernels = {k: {"ms": avg[k], "bytes": algo[k], "gbs": algo[k] / (avg[k] * 1e-3) / 1e9 if avg[k] > 0 else None,
                   "frac_hbm": algo[k] / (avg[k] * 1e-3) / 1e9 / peak if avg[k] > 0 else None} for k in avg}
    for k, ms in iso.items():
        kernels.setdefault(k, {"bytes": algo.get(k)})
        kernels[k]["isolated_ms"] = ms
        if kernels[k].get("bytes") and ms > 0:
            kernels[k]["gbs_isolated"] = kernels[k]["bytes"] / (ms * 1e-3) / 1e9
            kernels[k]["frac_hbm_isolated"] = kernels[k]["gbs_isolated"] / peak
    # the pages' per-unit formulas for the two big kernels: attention flops
    # (unmasked keys only) and the verifier's full-row byte count
    flops = attention_flops(w0)
    t_attn = avg["attention"]
    kernels["attention"]["tflops"] = flops / (t_attn * 1e-3) / 1e12 if t_attn > 0 else None
    kernels["attention"]["frac_tensor_burst"] = (kernels["attention"]["tflops"] / _bf16_peak()
                                                 if t_attn > 0 else None)
    n_int = sum(1 for b in range(w0.B) for u in range(int(w0.tree_off[b]), int(w0.tree_off[b + 1]))
                if any(int(w0.parent[c]) == u - int(w0.tree_off[b]) for c in range(u + 1, int(w0.tree_off[b + 1]))))
    full_rows = 4 * w0.V * (w0.T + (n_int if args.mode == "stochastic" else 0))
    kernels["verify"]["bytes_all_rows"] = full_rows
    kernels["verify"]["gbs_all_rows"] = full_rows / (avg["verify"] * 1e-3) / 1e9 if avg["verify"] > 0 else None
    # the walk is sequential in depth: its time per level of the deepest walk
    levels = max(1, int(passes[0].accept_len[:w0.B].max()))
    kernels["verify"]["levels"] = levels
    kernels["verify"]["us_per_level"] = 1e3 * avg["verify"] / levels
    if "isolated_ms" in kernels["verify"]:
        kernels["verify"]["us_per_level_isolated"] = 1e3 * kernels["verify"]["isolated_ms"] / levels
    achieved = kernels[dom]["gbs"]
    launches_per_step = 4 + (1 if _attn_splits(passes[0]) > 1 else 0) + (1 if _verify_uses_stats(w0, args.mode) else 0)
    traffic = _profiled_traffic(dom, args.mode, args.workload)

    # the dominant kernel's roof: tensor when its arithmetic intensity is above
    # the ridge point of the measured peaks (attention over wide trees), else HBM
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind}
    if dom == "attention" and t_attn > 0:
        ridge = _bf16_peak() * 1e12 / (peak * 1e9)
        if flops / algo["attention"] > ridge:
            tf = kernels["attention"]["tflops"]
            roofline = {"bound": "tensor", "kernel": dom, "achieved": tf, "peak": _bf16_peak(), "unit": "TFLOP/s",
                        "frac": tf / _bf16_peak(), "traffic": traffic, "peak_source": peak_kind + " (bf16 burst)",
                        "flop_per_byte": flops / algo["attention"], "ridge_flop_per_byte": ridge}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl["desc"], "verify": args.mode, "input_sets": n_sets,
                       "temperature": args.temperature, "draft_rows": "per child" if args.q_per_child else "per parent",
                       "l2": (f"{n_sets} rotating input sets of {_set_mb(works[0]):.0f} MB each (inputs larger than L2)"
                              if n_sets > 1 else f"one input set of {_set_mb(works[0]):.0f} MB (larger than L2)"),
                       "launch": "one CUDA graph per step (the C-ABI calls of the pass captured, no event nodes)",
                       "kernel_timing": "per kernel: ms = (K timed steps - the same K steps without that kernel) "
                                        "/ K, each run bracketed by CUDA events on the replay stream; isolated_ms = "
                                        "the kernel's call alone in a graph, L2 flushed before each replay, mean of "
                                        f"{ISO_REPLAYS} event-bracketed replays",
                       "tokens_per_step": tokens / args.steps / max(world, 1), "status_ok": status_ok,
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "clocks": clk.summary(),
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roofline,
            "kernels": kernels}
    if args.commit_layers > 0:
        line["commit_layers"] = measure_commit_layers(args.commit_layers, passes[0], dev)
    if args.tree_build:
        line["tree_build"] = measure_tree_build(dev)
    if args.dsd:
        line["dsd"] = measure_dsd(dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        workers = cpu_workers(works[0])
        pool = oracle_pool(workers)
        v, sample, _, used = run_cpu_baseline(works[0], args.mode, workers, pool)
        if pool is not None:
            pool.close()
            pool.join()
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _profiled_traffic(kernel, mode, workload=3):
    """DRAM bytes per launch (read + write) of the dominant kernel from the
    committed ncu figures (profiles/traffic.json), or None when there is no
    entry for this kernel, workload and mode, or the kernel source changed
    since the capture (the entry records the source's sha256 prefix)."""
    import hashlib
    src = {"attention": "attention_tc.cu", "verify": "verify.cu"}[kernel]
    path = os.path.join(ROOT, "tree_speculative_verification_spec_gb300", "csrc", src)
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entries = json.load(f)["entries"]
    except (OSError, ValueError, KeyError):
        return None
    for e in entries:
        if (e.get("kernel") == kernel and e.get("workload") == workload and e.get("mode") == mode
                and e.get("source_digest") == digest):
            return float(e["dram_bytes_per_launch"])
    return None


ISO_REPLAYS = 30


def isolated_times(vp, args, dev, stream, tree_kv):
    """Each call of one pass alone (input set 0): captured in its own graph,
    replayed ISO_REPLAYS times after 3 warm-up replays, with a write of twice
    the L2 size before every replay and CUDA events on the replay stream
    around the replay only.  Returns the mean milliseconds per call, by stage
    (attention includes its split-KV combine; stochastic verification its
    row statistics when it uses them; append is the tree K/V append)."""
    import torch
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(1, 2 * l2 // 4), dtype=torch.int32, device=dev)
    calls = {"mask": vp.mask_build, "append": lambda: vp.append(*tree_kv),
             "attention": lambda: vp.attention(args.attn_flags), "verify": lambda: vp.verify(args.mode),
             "commit": vp.commit}
    cap = torch.cuda.Stream(dev)
    out = {}
    for name, fn in calls.items():
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        torch.cuda.synchronize()
        for i in range(3):
            flush.fill_(i)
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ISO_REPLAYS)]
        for i, (a, b) in enumerate(ev):
            flush.fill_(i)
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        out[name] = sum(a.elapsed_time(b) for a, b in ev) / ISO_REPLAYS
        del g
    return out


def _verify_uses_stats(w, mode):
    """Whether the stochastic verifier launches its row-statistics kernel: the
    library does when the walk gets at most two CTAs per request (its cluster
    size: about one CTA per SM over the batch, wide enough for 16384-entry
    vocabulary slices)."""
    if mode != "stochastic":
        return False
    C = 1
    while C < 8 and w.B * C * 2 <= 152:
        C *= 2
    while C < 8 and (w.V + C - 1) // C > 16384:
        C *= 2
    return C <= 2


def _attn_splits(vp):
    import tree_speculative_verification_spec_gb300 as S
    b = vp.batch
    return 2 if S.spec_attention_workspace_size(b.B, b.T, b.n_max, b.max_prefix, b.Hq, b.Hkv, b.D) > 256 else 1


def _set_mb(w):
    """Bytes one pass reads from its input set (cache, queries, rows), in MB."""
    ts = (w.k_cache, w.v_cache, w.q, w.p_logits, w.q_probs)
    return sum(t.numel() * t.element_size() for t in ts) / 1e6


STEP_INPUTS = ("q", "parent", "tokens", "tree_off", "prefix_len", "p_logits", "q_probs", "uniforms")


def run_e2e(args, works, sets, passes, stream, dev, n_sets):
    """The pass through the C ABI with host buffers.  Every step copies its
    inputs (queries, tree arrays, the rows verification reads, and the tree's
    K/V rows) from pinned host memory into one of two device input slots (on a
    copy stream), appends the tree K/V after the prefix, runs the pass and
    reads its emitted tokens back; step i+1's copy overlaps step i's compute.
    The KV cache and block table are resident state, shared by the slots of
    one input set."""
    import dataclasses
    import torch
    from tree_speculative_verification_spec_gb300.pipeline import VerifyPass
    steps = max(3, args.steps)
    # the step's inputs: greedy verification reads neither draft rows nor uniforms
    names = [k for k in STEP_INPUTS if args.mode != "greedy" or k not in ("q_probs", "uniforms")]
    import workloads as W
    host, tree_host = [], []
    for j, w in enumerate(works):
        host.append({k: getattr(w, k).pin_memory() for k in names})
        # the tree's keys and values as the caller computes them: copied in and
        # appended after the prefix every step
        tree_host.append([t.pin_memory() for t in W.tree_kv_rows(w, 500 + j)])
    # two device slots per input set: the set's own buffers, and a shadow
    # with fresh per-step inputs and the same cache (and a pass of its own)
    slots = []
    for j in range(n_sets):
        d = sets[j]
        shadow = dataclasses.replace(d, **{k: torch.empty_like(getattr(d, k)) for k in names})
        vp2 = VerifyPass(shadow)
        vp2.inv_temp, vp2.q_layout = passes[j].inv_temp, passes[j].q_layout
        kv = [[torch.empty_like(t, device=dev) for t in tree_host[j]] for _ in range(2)]
        slots.append([(d, passes[j], kv[0]), (shadow, vp2, kv[1])])
    out_tok = [[torch.empty((p.batch.B, p.batch.n_max), dtype=torch.int32).pin_memory() for _ in range(2)]
               for p in passes]
    out_n = [[torch.empty(p.batch.B, dtype=torch.int32).pin_memory() for _ in range(2)] for p in passes]
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    h2d += sum(t.numel() * t.element_size() for t in tree_host[0])
    d2h = out_tok[0][0].numel() * 4 + out_n[0][0].numel() * 4
    copy_stream = torch.cuda.Stream(dev)
    copied = [[torch.cuda.Event() for _ in range(2)] for _ in range(n_sets)]
    consumed = [[torch.cuda.Event() for _ in range(2)] for _ in range(n_sets)]
    used = [[False, False] for _ in range(n_sets)]

    def e2e_step(i):
        j, k = i % n_sets, (i // n_sets) % 2
        d, vp, kv = slots[j][k]
        h = host[j]
        with torch.cuda.stream(copy_stream):
            if used[j][k]:
                copy_stream.wait_event(consumed[j][k])  # the slot's previous pass has read its inputs
            for name, t in h.items():
                getattr(d, name).copy_(t, non_blocking=True)
            for dst, src in zip(kv, tree_host[j]):
                dst.copy_(src, non_blocking=True)
            copied[j][k].record(copy_stream)
        stream.wait_event(copied[j][k])
        vp.run(args.mode, args.attn_flags, tree_kv=kv)
        consumed[j][k].record(stream)
        used[j][k] = True
        out_tok[j][k].copy_(vp.emitted, non_blocking=True)
        out_n[j][k].copy_(vp.n_emitted, non_blocking=True)
        return j, k

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    done = []
    for i in range(steps):
        done.append(e2e_step(i))
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    # every step's result was read back inside the timed region; a slot's
    # inputs are the same at every step, so its last read-back counts for all
    per_slot = {(j, k): int(out_n[j][k].sum()) for j in range(n_sets) for k in range(2)}
    toks = sum(per_slot[jk] for jk in done)
    # whole job: the slowest rank's time, the tokens of all ranks (copies per rank)
    ms, toks = aggregate_replicas(ms, float(toks), dev)
    world = _dist()[0]
    return {"value": toks / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d * world,
            "d2h_bytes_per_step": d2h * world,
            "ms_per_step": ms / steps,
            "overlap": "step i+1's host-to-device copy (copy stream) overlaps step i's pass; two input slots",
            "pass": "mask build, tree K/V append (rows copied from the host), attention, verification, commit"}


def measure_commit_layers(L, vp, dev, reps=20, replays=5):
    """The commit of L layers' caches for input set 0 in one launch, against L
    single-layer launches, and the layered commit followed by the page release
    (the block table and the pool count put back before each, and that reset
    timed alone and subtracted).  Each figure: one graph of `reps` back-to-back
    calls, replayed `replays` times between CUDA events; microseconds per call."""
    import torch
    import tree_speculative_verification_spec_gb300 as S
    d = vp.batch
    ks = [d.k_cache] + [torch.empty_like(d.k_cache) for _ in range(L - 1)]
    vs = [d.v_cache] + [torch.empty_like(d.v_cache) for _ in range(L - 1)]
    kp = torch.tensor([t.data_ptr() for t in ks], dtype=torch.int64, device=dev)
    vp_ = torch.tensor([t.data_ptr() for t in vs], dtype=torch.int64, device=dev)
    dtype = S.SPEC_BF16 if d.k_cache.element_size() == 2 else S.SPEC_F32
    new_len = torch.zeros(d.B, dtype=torch.int32, device=dev)
    st = torch.zeros(d.B, dtype=torch.int32, device=dev)
    bt0 = d.block_table.clone()
    pool = torch.empty(d.B * d.max_blocks, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)

    def layered(release):
        S.spec_kv_commit_layers(kp, vp_, L, d.block_table, d.max_blocks, d.block_size, d.num_blocks, d.prefix_len,
                                d.tree_off, vp.path, d.n_max, vp.accept_len, d.B, d.Hkv, d.D, dtype, new_len,
                                pool if release else None, cnt if release else None, st)

    def per_layer():
        for l in range(L):
            S.spec_kv_commit(ks[l], vs[l], d.block_table, d.max_blocks, d.block_size, d.num_blocks, d.prefix_len,
                             vp.path, d.n_max, vp.accept_len, d.B, d.Hkv, d.D, new_len, st)

    def reset():
        d.block_table.copy_(bt0)
        cnt.zero_()

    def with_release():
        reset()
        layered(True)

    def time_us(fn):
        cap = torch.cuda.Stream(dev)
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for _ in range(reps):
                fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream(dev)
        a.record(stream)
        for _ in range(replays):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * replays)

    one = time_us(lambda: layered(False))
    many = time_us(per_layer)
    rel = time_us(with_release) - time_us(reset)
    with_release()
    torch.cuda.synchronize()
    released = int(cnt.item())
    reset()
    torch.cuda.synchronize()
    ok = int(st.abs().sum()) == 0
    return {"layers": L, "us_one_launch": one, "us_per_layer_launches": many, "us_commit_and_release": rel,
            "pages_released": released, "status_ok": ok}


def measure_tree_build(dev, reps=20, replays=5):
    """Device tree construction on the decode layer's shapes: the expansion
    schedule <4,2,2,1,1,1,1,1> (8 requests, V = 32000, every level's draft rows
    resident; three rotating row sets, 285 MB together, above L2), and the
    merge of 32 candidate sequences of 8 tokens per request for 64 requests.
    Each: one graph of `reps` builds, replayed `replays` times between CUDA
    events; microseconds per build."""
    import torch
    import tree_speculative_verification_spec_gb300 as S
    B, V, sched = 8, 32000, [4, 2, 2, 1, 1, 1, 1, 1]
    sizes = [1]
    for k in sched:
        sizes.append(sizes[-1] * k)
    n_total = sum(sizes)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    sets = [[torch.randn((B * sizes[lev], V), generator=g, device=dev) for lev in range(len(sched))]
            for _ in range(3)]
    roots = torch.randint(0, V, (B,), generator=g, device=dev, dtype=torch.int32)
    tree_off = torch.empty(B + 1, dtype=torch.int32, device=dev)
    par = torch.empty(B * n_total, dtype=torch.int32, device=dev)
    tok = torch.empty(B * n_total, dtype=torch.int32, device=dev)

    def expand(rows):
        S.spec_tree_init(roots, B, n_total, tree_off, par, tok)
        start = 0
        for lev, k in enumerate(sched):
            S.spec_tree_expand_level(rows[lev], B, sizes[lev], V, k, start, n_total, par, tok)
            start += sizes[lev]

    Bm, M, m = 64, 32, 8
    seqs = torch.randint(0, 6, (Bm, M, m), generator=g, device=dev, dtype=torch.int32)  # shared prefixes
    lens = torch.full((Bm, M), m, dtype=torch.int32, device=dev)
    mroots = torch.zeros(Bm, dtype=torch.int32, device=dev)
    cap = Bm * (1 + M * m)
    moff = torch.empty(Bm + 1, dtype=torch.int32, device=dev)
    mpar, mtok, msrc = (torch.empty(cap, dtype=torch.int32, device=dev) for _ in range(3))
    mnode = torch.empty(Bm * M * m, dtype=torch.int32, device=dev)
    mst = torch.empty(Bm, dtype=torch.int32, device=dev)

    def merge():
        S.spec_tree_merge(seqs, lens, mroots, Bm, M, m, 32000, moff, mpar, mtok, msrc, mnode, mst)

    def time_us(fns):
        cap_s = torch.cuda.Stream(dev)
        for f in fns:
            f()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap_s):
            for r in range(reps):
                fns[r % len(fns)]()
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream(dev)
        a.record(stream)
        for _ in range(replays):
            gr.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * replays)

    t_exp = time_us([lambda r=r: expand(r) for r in sets])
    t_merge = time_us([merge])
    rows_bytes = sum(B * sizes[lev] * V * 4 for lev in range(len(sched)))
    peak, _ = _peaks()
    gbs = rows_bytes / (t_exp * 1e-6) / 1e9
    return {"expansion": {"schedule": sched, "requests": B, "V": V, "nodes_per_tree": n_total,
                          "us_per_build": t_exp, "launches": 1 + len(sched), "row_bytes": rows_bytes,
                          "gbs": gbs, "frac_hbm": gbs / peak},
            "merge": {"requests": Bm, "sequences": M, "tokens_per_sequence": m, "us_per_build": t_merge,
                      "launches": 3, "nodes": int(moff[-1].item())}}


def measure_dsd(dev, bss=(1, 4, 16, 64, 256), max_k=8, replays=20):
    """Offline goodput profile of this pass ("Hardware-aware dynamic
    speculative decoding"): for each batch size, the sweep workload's chains
    (prefix 4096, V = 32000, alpha = 0.3) cut to K + 1 nodes for K = 1..max_k;
    each <tokens = B (K + 1), K> pass captured once in the graph cache and
    replayed; ITL = the replay time (this library's verification pass:
    mask, one attention layer, verification, commit); AL = emitted tokens per
    request, averaged over the largest batch (acceptance is a property of the
    draft/target pair, not of the batch size; one request alone is too few).
    The table's optimal K per batch size comes from the library.  Beside the
    measured AL: the closed form (1 - a^(K+1)) / (1 - a) of "Inference
    Optimization Techniques" with a = the mean over the drafts of
    sum_x min(p(x), q(x)) (the per-draft acceptance probability), computed on
    the host from the largest batch's rows."""
    import torch
    import workloads as W
    from tree_speculative_verification_spec_gb300.dynamic_k import DynamicK, GraphCache
    from tree_speculative_verification_spec_gb300.pipeline import DeviceBatch, VerifyPass
    ks = list(range(1, max_k + 1))
    pol = DynamicK(bss, ks)
    itl, al_big = {}, {}
    for i, B in enumerate(bss):
        full = W.config4(K=max_k, B=B, tree="chain", alpha=0.3)
        made = {}

        def make(tokens, K):
            vp = VerifyPass(DeviceBatch.from_workload(W.chain_prefix(full, K + 1), device=dev))
            made[(tokens, K)] = vp
            return vp

        cache = GraphCache(make)
        for j, K in enumerate(ks):
            key = (B * (K + 1), K)
            vp = cache.replay(*key)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            stream = torch.cuda.current_stream(dev)
            a.record(stream)
            for _ in range(replays):
                cache.replay(*key)
            b.record(stream)
            torch.cuda.synchronize()
            itl[(i, j)] = a.elapsed_time(b) * 1e3 / replays
            if B == max(bss):
                al_big[j] = float(vp.n_emitted[:B].float().mean())
        if B == max(bss):
            # per-draft acceptance: rows of the chains' parents (nodes 0 .. max_k - 1)
            rows = torch.cat([torch.arange(b * (max_k + 1), b * (max_k + 1) + max_k) for b in range(B)])
            p = torch.softmax(full.p_logits[rows].double(), -1)
            a_hat = float(torch.minimum(p, full.q_probs[rows].double()).sum(-1).mean())
        del cache, made, full
        torch.cuda.empty_cache()
    for (i, j), t in itl.items():
        pol.record(i, j, al_big[j], t)
    k_opt = pol.optimal_k()
    closed = [(1 - a_hat ** (K + 1)) / (1 - a_hat) for K in ks]
    return {"batch_sizes": list(bss), "k_values": ks, "acceptance_a": a_hat,
            "al_measured": [round(al_big[j], 4) for j in range(len(ks))],
            "al_closed_form": [round(x, 4) for x in closed],
            "al": [[round(x, 4) for x in r] for r in pol.al.tolist()],
            "itl_us": [[round(x, 2) for x in r] for r in pol.itl.tolist()],
            "goodput_tok_per_us": [[round(a / t, 5) for a, t in zip(ra, rt)] for ra, rt in zip(pol.al, pol.itl)],
            "k_opt": k_opt.tolist(), "graphs_captured": len(bss) * len(ks)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--mode", default=None, choices=["stochastic", "greedy"])
    ap.add_argument("--workload", type=int, default=3, choices=sorted(WORKLOADS))
    ap.add_argument("--attn-flags", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0, help="offset added to the workload's input seeds")
    ap.add_argument("--temperature", type=float, default=None,
                    help="stochastic verification at this temperature for every request (default: none, T = 1)")
    ap.add_argument("--q-per-child", action="store_true",
                    help="read the draft rows per child (merged trees) instead of per parent")
    ap.add_argument("--tree-build", action="store_true", help="also time device tree construction")
    ap.add_argument("--dsd", action="store_true", help="also profile goodput = AL / ITL per batch size and K")
    ap.add_argument("--commit-layers", type=int, default=0,
                    help="also time the commit of this many layers' caches in one launch (0: off)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.mode is None:
        args.mode = WORKLOADS[args.workload]["mode"]
    if args.impl == "reference":
        return bench_reference(args)
    return bench_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
