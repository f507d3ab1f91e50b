#!/usr/bin/env python
"""DSA decode-layer benchmark: indexer -> top-k -> sparse MLA -> merge.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long_128k]

Prints ONE JSON line (rank 0).  A step is one pass of the whole decode layer
over one synthetic batch (default: 8 requests x 131072 cached tokens, one
query token each, k = 2048, 128 MLA heads), inputs resident in HBM.  A step
is one dsa_decode_fused call (workspace clear and the four kernels).  The K
timed steps run back to back as the layers of a decode step do, each on its
own copy of the inputs (8 copies in turn, so no step finds its inputs in L2;
no flush), from CUDA graphs of up to 64 calls; one pair of CUDA events on the
launching stream brackets all K.  For comparison the line also gives the
median of steps run one per graph replay with L2 flushed before each (each
then also pays the replay's launch).  A separate pass through the library's timed entry
point (an event before each kernel) gives the per-stage times and the
dominant kernel's (the indexer's) duration for the roofline.  `--impl reference` times the float64 CPU oracle on
a bounded sample of the same workload.

Multi-GPU (torchrun): one process per GPU, each runs its own batch (requests
are independent; no data-path collective); value = all ranks' query tokens /
the slowest rank's time.
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

METRIC = "DSA decode layer µs and tokens/s at 128K ctx, k=2048; achieved HBM GB/s vs 8 TB/s"
UNIT = "query-tokens/s"
TARGET_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
NCOPY = 8   # input copies a timed sequence of layers cycles through


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="long_128k")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-configuration table (other workloads)")
    p.add_argument("--copies", type=int, default=NCOPY,
                   help="input copies the timed layers cycle through (1: every layer on the same "
                        "inputs, for profiling with a small device footprint)")
    return p.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def indexer_traffic(workload: str):
    """DRAM bytes per indexer launch from the committed ncu summary, if that
    summary was taken on the current indexer source."""
    src = os.path.join(ROOT, "deepseek_sparse_attention_lightning_gb300", "csrc", "indexer.cu")
    summ = os.path.join(ROOT, "profiles", f"indexer_{workload}.md")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        fields = {}
        for line in open(summ):
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
        if fields.get("indexer_cu_sha256") != sha:
            return None
        return float(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    """Maximum of ``x`` over the ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(tokens_per_step: int, steps: int, world: int, total_ms_max: float) -> float:
    """Whole-job query tokens per second: every rank ran ``steps`` steps of
    ``tokens_per_step`` query tokens; the job took the slowest rank's time."""
    return tokens_per_step * steps * world / (total_ms_max / 1e3)


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def accounting(spec, seqlens):
    """Algorithmic bytes/FLOPs of one decode layer: index keys (128 FP8 B +
    4 B scale per cached token, read once per request) + gathered latent rows
    (1152 B per selected token per query); FLOPs 16384 per (query, visible key)
    in the indexer and 2H*576 + 2H*512 per (query, selected key) in MLA."""
    nq, k, H = spec.q_per_req, spec.topk, spec.num_heads
    idx_bytes = sum(int(s) * 132 for s in seqlens)
    sel = 0
    vis_total = 0
    for s in seqlens:
        for i in range(nq):
            v = max(int(s) - (nq - 1 - i), 0)
            vis_total += v
            sel += min(v, k)
    att_bytes = sel * 1152
    return dict(query_tokens=len(seqlens) * nq, layer_bytes=idx_bytes + att_bytes,
                indexer_bytes=idx_bytes, attention_bytes=att_bytes,
                indexer_flops=vis_total * 16384, attention_flops=sel * (2 * H * 576 + 2 * H * 512))


# ---------------------------------------------------------------------------
# CPU (oracle) leg
# ---------------------------------------------------------------------------

class OracleSampler:
    """Times the float64 oracle on whole requests of the workload, one request
    at a time with its data already in host memory (each request's inputs are
    prepared once, outside the timed part), cycling over the requests."""

    def __init__(self, wl):
        import numpy as np
        self.wl, self.np = wl, np
        self.seqlens = wl.seqlens.cpu().numpy()
        self.table = wl.page_table.cpu().numpy()
        self.prepared = {}
        self.cursor = 0

    def _inputs(self, r):
        if r in self.prepared:
            return self.prepared[r]
        import torch
        import oracle as O
        from deepseek_sparse_attention_lightning_gb300 import workloads as W
        np, wl, spec = self.np, self.wl, self.wl.spec
        nq = spec.q_per_req
        S = int(self.seqlens[r])
        rows = torch.from_numpy(O.physical_rows(self.table[r], np.arange(S))).to(wl.k_fp8.device)
        t0, t1 = r * nq, (r + 1) * nq
        inputs = dict(
            seqlens=np.array([S]), page_table=np.arange((S + 63) // 64)[None, :], q_per_req=nq,
            q_fp8=wl.q_fp8[t0:t1].cpu().numpy(), q_scale=wl.q_scale[t0:t1].cpu().numpy(),
            w=wl.w[t0:t1].cpu().numpy(), k_fp8=wl.k_fp8[rows].cpu().numpy(),
            k_scale=wl.k_scale[rows].cpu().numpy(), q=W.bf16_bits(wl.q[t0:t1]),
            kv=W.bf16_bits(wl.kv[rows]), sm_scale=spec.sm_scale, topk=spec.topk)
        pad = (-S) % 64
        if pad:
            inputs["k_fp8"] = np.concatenate([inputs["k_fp8"], np.zeros((pad, 128), np.uint8)])
            inputs["k_scale"] = np.concatenate([inputs["k_scale"], np.ones(pad, np.float32)])
            inputs["kv"] = np.concatenate([inputs["kv"], np.zeros((pad, 576), np.uint16)])
        self.prepared[r] = inputs
        return inputs

    def sample(self, seconds: float):
        """Whole requests (at least one) until ``seconds`` of oracle time:
        (query rows, seconds spent, requests)."""
        import oracle as O
        spec = self.wl.spec
        rows, spent, requests = 0, 0.0, 0
        while requests == 0 or spent < seconds:
            inputs = self._inputs(self.cursor % spec.batch)
            self.cursor += 1
            start = time.perf_counter()
            O.decode_layer(inputs)
            spent += time.perf_counter() - start
            rows += spec.q_per_req
            requests += 1
        return rows, spent, requests


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


class OneCore:
    """Pins every thread of this process (BLAS workers included) to one of
    its cores for the duration of a `with` block, then restores each thread's
    affinity: the oracle then runs on a single core."""

    def __enter__(self):
        self.saved = {}
        try:
            allowed = sorted(os.sched_getaffinity(0))
            self.core = allowed[0]
            for tid in os.listdir("/proc/self/task"):
                t = int(tid)
                try:
                    self.saved[t] = os.sched_getaffinity(t)
                    os.sched_setaffinity(t, {self.core})
                except OSError:
                    pass
            self.ok = True
        except (AttributeError, OSError):
            self.ok = False
        return self

    def __exit__(self, *exc):
        for t, cpus in self.saved.items():
            try:
                os.sched_setaffinity(t, cpus)
            except OSError:
                pass
        return False


def run_reference(args, world, rank):
    if rank != 0:
        return
    import torch
    from deepseek_sparse_attention_lightning_gb300 import workloads as W
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = W.make_workload(args.workload, device=dev)
    units = accounting(wl.spec, wl.seqlens.cpu().tolist())
    per_step = []
    rows = 0
    # each step a bounded sample (at least one whole request), the whole run
    # about --cpu-seconds of oracle time beyond one request per step
    sampler = OracleSampler(wl)
    budget = args.cpu_seconds / max(1, args.steps + args.warmup)
    for i in range(args.warmup + args.steps):
        n, spent, nreq = sampler.sample(budget)
        if i >= args.warmup:
            per_step.append(spent / n)
            rows += n
    sec_per_row = sum(per_step) / len(per_step)
    value = 1.0 / sec_per_row
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec_per_row * 1e3 * units["query_tokens"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": wl.spec.batch, "q_per_req": wl.spec.q_per_req,
                   "seqlen": wl.spec.seqlen, "topk": wl.spec.topk, "heads": wl.spec.num_heads},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{rows} query rows (whole requests, one at a time) of the "
                                   f"{args.workload} workload, float64 numpy oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

def pctl(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, int(q * len(xs)))]


def clone_workload(W, wl):
    """The same workload in new device memory: every layer of a model reads
    its own caches, so a run of layers cycling through NCOPY such copies
    finds none of a layer's inputs in L2 (8 x ~160 MB touched in between)."""
    import dataclasses
    return dataclasses.replace(
        wl, seqlens=wl.seqlens.clone(), page_table=wl.page_table.clone(), q_fp8=wl.q_fp8.clone(),
        q_scale=wl.q_scale.clone(), w=wl.w.clone(),
        layers=[W.LayerCache(lc.k_fp8.clone(), lc.k_scale.clone(), lc.q.clone(), lc.kv.clone())
                for lc in wl.layers])


def time_layer_sequence(torch, fns, steps, sampler=None, barrier=None):
    """Time `steps` layer calls run back to back as in a decode step: call j
    is fns[j % len(fns)] (each on its own copy of the inputs), captured into
    CUDA graphs of up to 64 calls; one event pair brackets all of them.
    Returns (total ms, how it was timed)."""
    G = max(1, min(steps, 64))
    nfull, rem = divmod(steps, G)

    def cap(n):
        if n == 0:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(n):
                fns[j % len(fns)]()
        torch.cuda.synchronize()
        return g

    try:
        gfull, grem = cap(G), cap(rem)
        how = f"CUDA graphs of {G} back-to-back layer calls, replayed"
    except Exception as exc:  # noqa: BLE001 -- reported in the JSON line
        torch.cuda.synchronize()
        gfull = grem = None
        how = "direct calls (graph capture failed: " + f"{type(exc).__name__}: {exc}"[:160] + ")"

    def run(n_full, with_rem):
        if gfull is None:
            for j in range(n_full * G + (rem if with_rem else 0)):
                fns[j % len(fns)]()
            return
        for _ in range(n_full):
            gfull.replay()
        if with_rem and grem is not None:
            grem.replay()

    # untimed load first: the clocks are sampled under load, the caches and
    # TLBs see the same cycle of copies as the timed run
    if sampler is not None:
        sampler.start()
    t_end = time.time() + 0.3
    while time.time() < t_end:
        run(1, False)
        torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)   # keep the host ahead: every replay is queued before e0 fires
    e0.record()
    run(nfull, True)
    e1.record()
    torch.cuda.synchronize()
    if barrier is not None:
        barrier()
    return e0.elapsed_time(e1), how


def measure_configs(torch, api, W, dev, steps):
    """The other workloads of the benchmark table, each timed like the
    headline (a run of back-to-back layer calls cycling through NCOPY copies
    of the inputs, from CUDA graphs, one event pair around the run):
    tiny_4k cold and warm (warm: one copy, so its inputs stay in L2),
    mtp_32k, long_varlen, short_dense as the DSA layer and as the dense path
    (the same attention over every visible token, given as the selection),
    and mli_195k's two layers serial vs the second layer through
    dsa_decode_mli (its attention reuses the first layer's selection while
    its own indexer + top-k run beside it); the new tokens' cache write alone (*_cache_write) and fused
    in front of the layer (*_with_cache_write); long_128k and mtp_32k with
    the latent cache in FP8 (*_fp8_latent)."""
    res = {}

    def timed(make_fn, wls, n):
        fns = [make_fn(c) for c in wls]
        for f in fns:
            f()
        torch.cuda.synchronize()
        total_ms, how = time_layer_sequence(torch, fns, n)
        if api.dsa_get_device_error() != 0:
            raise RuntimeError("device error while timing a configuration")
        t = {"us_per_step": total_ms / n * 1e3}
        if not how.startswith("CUDA graphs"):
            t["timing"] = how   # a fallback to direct calls times the host's launches too
        return t

    def layer_fn(wl, layer=0, topk_in=None, topk_out=None, ws=None, out=None):
        spec = wl.spec
        desc = api.workload_desc(wl)
        splits = api.dsa_num_splits_auto(desc)
        msl = wl.max_seqlen
        ws = api.alloc_workspace(wl, splits) if ws is None else ws
        out = torch.empty((spec.num_tokens, spec.num_heads, 512), dtype=torch.float32, device=dev) \
            if out is None else out
        lc = wl.layers[layer]

        def fn():
            api.dsa_decode_fused(desc, wl.q_fp8, wl.q_scale, wl.w, lc.k_fp8, lc.k_scale, lc.q, lc.kv,
                                 out, ws, msl, spec.sm_scale, splits, topk_in, topk_out,
                                 stream=torch.cuda.current_stream())
        return fn

    def record(name, wl, t, layers=1):
        u = accounting(wl.spec, wl.seqlens.cpu().tolist())
        us = t["us_per_step"]
        t.update(query_tokens_per_s=u["query_tokens"] / (us * 1e-6),
                 layer_bytes=layers * u["layer_bytes"],
                 layer_gbs=layers * u["layer_bytes"] / (us * 1e-6) / 1e9,
                 frac_of_8tbs=layers * u["layer_bytes"] / (us * 1e-6) / 1e9 / TARGET_HBM_GBS)
        res[name] = t

    n = max(24, min(steps, 200))
    for name in ("tiny_4k", "mtp_32k", "long_varlen", "short_dense", "mli_195k"):
        wl = W.make_workload(name, device=dev)
        copies = [wl] + [clone_workload(W, wl) for _ in range(NCOPY - 1)]
        # one workspace and output for all copies, as a model reuses them
        ws0 = api.alloc_workspace(wl, api.dsa_num_splits_auto(api.workload_desc(wl)))
        out0 = torch.empty((wl.spec.num_tokens, wl.spec.num_heads, 512), dtype=torch.float32,
                           device=dev)

        def plain(c, **kw):
            return layer_fn(c, ws=ws0, out=out0, **kw)

        def cache_write(c):
            # the step before the indexer: the new tokens' latent rows and
            # FP8 indexer keys written into the caches (same rows every call)
            T = c.spec.num_tokens
            gen = torch.Generator(device=dev).manual_seed(1)
            lat = torch.randn(T, 576, generator=gen, device=dev).to(torch.bfloat16)
            key = torch.randn(T, 128, generator=gen, device=dev).to(torch.bfloat16)
            cdesc = api.workload_desc(c)

            def fn():
                api.dsa_cache_write(cdesc, lat, key, c.kv, c.k_fp8, c.k_scale,
                                    stream=torch.cuda.current_stream())
            return fn

        def fused_write(c):
            # the cache write and the layer in one call (dsa_decode_fused_write)
            T, spec = c.spec.num_tokens, c.spec
            gen = torch.Generator(device=dev).manual_seed(1)
            lat = torch.randn(T, 576, generator=gen, device=dev).to(torch.bfloat16)
            key = torch.randn(T, 128, generator=gen, device=dev).to(torch.bfloat16)
            cdesc = api.workload_desc(c)
            splits = api.dsa_num_splits_auto(cdesc)
            lc, msl = c.layers[0], c.max_seqlen

            def fn():
                api.dsa_decode_fused_write(cdesc, lat, key, c.q_fp8, c.q_scale, c.w, lc.k_fp8,
                                           lc.k_scale, lc.q, lc.kv, out0, ws0, msl,
                                           spec.sm_scale, splits,
                                           stream=torch.cuda.current_stream())
            return fn

        if name != "mli_195k":
            t = timed(cache_write, copies, n)
            T = wl.spec.num_tokens
            t.update(rows=T, bytes=T * (2 * 576 * 2 + 128 * 2 + 128 + 4),
                     note="latent rows + FP8 index keys of the new tokens; launch-bound")
            res[name + "_cache_write"] = t
            if name != "tiny_4k":
                record(name + "_with_cache_write", wl, timed(fused_write, copies, n))
        if name == "tiny_4k":
            record(name, wl, timed(plain, copies, n))
            record(name + "_warm", wl, timed(plain, [wl], n))
        elif name == "short_dense":
            record(name, wl, timed(plain, copies, n))
            # dense path: every visible position given as the selection
            T, k = wl.spec.num_tokens, wl.spec.topk
            vis = [max(int(s), 0) for s in wl.seqlens.cpu().tolist()]
            ident = torch.full((T, k), -1, dtype=torch.int32)
            for t, v in enumerate(vis):
                ident[t, :min(v, k)] = torch.arange(min(v, k), dtype=torch.int32)
            ident = ident.to(dev)
            r = timed(lambda c: plain(c, topk_in=ident), copies, n)
            record(name + "_dense", wl, r)
            res[name]["overhead_vs_dense_us"] = res[name]["us_per_step"] - r["us_per_step"]
        elif name == "mli_195k":
            T, k = wl.spec.num_tokens, wl.spec.topk
            sel1 = torch.empty((T, k), dtype=torch.int32, device=dev)
            sel2 = torch.empty((T, k), dtype=torch.int32, device=dev)

            def serial(c):
                f1, f2 = plain(c, layer=0, topk_out=sel1), plain(c, layer=1)

                def fn():
                    f1()
                    f2()
                return fn

            def overlapped(c):
                # layer 1 as usual; layer 2 through dsa_decode_mli: its
                # attention over layer 1's selection, its own indexer + top-k
                # on the SMs the attention leaves free
                f1 = plain(c, layer=0, topk_out=sel1)
                desc, lc2, spec = api.workload_desc(c), c.layers[1], c.spec
                msl = c.max_seqlen

                def fn():
                    f1()
                    api.dsa_decode_mli(desc, c.q_fp8, c.q_scale, c.w, lc2.k_fp8, lc2.k_scale,
                                       lc2.q, lc2.kv, sel1, sel2, out0, ws0, msl, spec.sm_scale,
                                       stream=torch.cuda.current_stream())
                return fn

            a = timed(serial, copies, n)
            b = timed(overlapped, copies, n)
            record("mli_195k_serial_2layers", wl, a, layers=2)
            record("mli_195k_overlapped_2layers", wl, b, layers=2)
            res["mli_195k_overlapped_2layers"]["speedup_vs_serial"] = a["us_per_step"] / b["us_per_step"]
        else:
            record(name, wl, timed(plain, copies, n))
        del wl, copies, ws0, out0
        torch.cuda.empty_cache()
    # The layer over an FP8 latent cache (656-byte rows: dsa_decode_fused_fp8kv)
    # on the long-context workloads; the bf16 layer of the same workload is
    # the headline (long_128k) or the entry above (mtp_32k).
    for name in ("long_128k", "mtp_32k"):
        wl = W.make_workload(name, device=dev)
        copies = [wl] + [clone_workload(W, wl) for _ in range(NCOPY - 1)]
        ws0 = api.alloc_workspace(wl, api.dsa_num_splits_auto(api.workload_desc(wl)))
        out0 = torch.empty((wl.spec.num_tokens, wl.spec.num_heads, 512), dtype=torch.float32,
                           device=dev)
        kv8s = []
        for c in copies:
            kv = c.layers[0].kv
            kv8 = torch.empty((kv.shape[0], 656), dtype=torch.uint8, device=dev)
            api.dsa_latent_to_fp8(kv, kv8)
            kv8s.append(kv8)

        def fp8_layer(i):
            c, kv8, spec = copies[i], kv8s[i], copies[i].spec
            cdesc = api.workload_desc(c)
            splits = api.dsa_num_splits_auto(cdesc)
            lc, msl = c.layers[0], c.max_seqlen

            def fn():
                api.dsa_decode_fused_fp8kv(cdesc, c.q_fp8, c.q_scale, c.w, lc.k_fp8, lc.k_scale,
                                           lc.q, kv8, out0, ws0, msl, spec.sm_scale, splits,
                                           stream=torch.cuda.current_stream())
            return fn

        t = timed(fp8_layer, list(range(len(copies))), n)
        u = accounting(wl.spec, wl.seqlens.cpu().tolist())
        fp8_bytes = u["indexer_bytes"] + (u["attention_bytes"] // 1152) * 656
        us = t["us_per_step"]
        t.update(query_tokens_per_s=u["query_tokens"] / (us * 1e-6), layer_bytes=fp8_bytes,
                 layer_gbs=fp8_bytes / (us * 1e-6) / 1e9,
                 frac_of_8tbs=fp8_bytes / (us * 1e-6) / 1e9 / TARGET_HBM_GBS,
                 note="latent cache in FP8 rows of 656 B (gathered bytes 656 per selected token)")
        res[name + "_fp8_latent"] = t
        del copies, kv8s, wl
        torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    import torch
    from deepseek_sparse_attention_lightning_gb300 import api, build
    from deepseek_sparse_attention_lightning_gb300 import workloads as W

    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.make_workload(args.workload, device=dev)
    spec = wl.spec
    seqlens = wl.seqlens.cpu().tolist()
    units = accounting(spec, seqlens)
    T, H, k = spec.num_tokens, spec.num_heads, spec.topk
    desc = api.workload_desc(wl)
    splits = api.dsa_num_splits_auto(desc)
    ws = api.alloc_workspace(wl, splits)
    out = torch.empty((T, H, 512), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    max_seqlen = wl.max_seqlen      # read once: a device read cannot sit in a graph capture

    def layer(stage_events=None):
        api.dsa_decode_fused(desc, wl.q_fp8, wl.q_scale, wl.w, wl.k_fp8, wl.k_scale, wl.q, wl.kv,
                             out, ws, max_seqlen, spec.sm_scale, splits,
                             stream=torch.cuda.current_stream(), stage_events=stage_events)

    def make_events(n, m):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(m)] for _ in range(n)]
        for row in ev:      # create the events (torch creates them lazily on record)
            for e in row:
                e.record()
        return ev

    def capture(fn):
        """The layer call captured once into a CUDA graph (None if capture
        fails, e.g. on a driver without it; steps then call the library)."""
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            torch.cuda.synchronize()
            return g
        except Exception as exc:  # noqa: BLE001 -- reported in the JSON line
            capture_errors.append(f"{type(exc).__name__}: {exc}"[:200])
            torch.cuda.synchronize()
            return None

    capture_errors = []

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        layer()
    torch.cuda.synchronize()
    if api.dsa_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # A step is one dsa_decode_fused call (workspace clear + four kernels).
    # The K timed steps run back to back, as the layers of a decode step do,
    # each on its own copy of the inputs (NCOPY copies in turn, so no step
    # finds its inputs in L2), from CUDA graphs; one event pair brackets all
    # K steps.
    copies = [wl] + [clone_workload(W, wl) for _ in range(max(1, args.copies) - 1)]

    def layer_on(c):
        cdesc = api.workload_desc(c)

        def fn():
            api.dsa_decode_fused(cdesc, c.q_fp8, c.q_scale, c.w, c.k_fp8, c.k_scale, c.q, c.kv,
                                 out, ws, max_seqlen, spec.sm_scale, splits,
                                 stream=torch.cuda.current_stream())
        return fn

    K = args.steps
    sampler = ClockSampler(local)
    total_ms, timed_how = time_layer_sequence(torch, [layer_on(c) for c in copies], K,
                                              sampler=sampler, barrier=lambda: dist_barrier(world))
    clocks = sampler.stop()
    if api.dsa_get_device_error() != 0:
        raise RuntimeError("device error during the timed steps")

    # For comparison: one layer per graph replay with L2 flushed before each
    # (the flush outside the events), so each step also pays the graph's
    # launch; median over up to 300 steps.
    graph = capture(layer)
    KP = max(1, min(K, 300))
    ev = make_events(KP, 2)
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)
    for i in range(KP):
        flush.zero_()
        ev[i][0].record()
        if graph is not None:
            graph.replay()
        else:
            layer()
        ev[i][1].record()
    torch.cuda.synchronize()
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(KP)]

    # Stage breakdown, a separate pass: the layer with an event before each
    # kernel, read back after every step (a device sleep first keeps the host
    # ahead, so no stage waits on a launch).  Events between kernels keep each
    # launch from overlapping the tail of the one before, so these stages add
    # up to more than a timed step.
    sev = make_events(1, 5)[0]
    KS = max(1, min(K, 300))
    idx_ms, topk_ms, mla_ms, merge_ms = [], [], [], []
    for i in range(KS):
        torch.cuda._sleep(400_000)
        flush.zero_()
        layer(sev)
        torch.cuda.synchronize()
        idx_ms.append(sev[0].elapsed_time(sev[1]))
        topk_ms.append(sev[1].elapsed_time(sev[2]))
        mla_ms.append(sev[2].elapsed_time(sev[3]))
        merge_ms.append(sev[3].elapsed_time(sev[4]))
    total_ms_max = dist_max(total_ms, world)
    ms_per_step = total_ms_max / K
    value = throughput(units["query_tokens"], K, world, total_ms_max)

    # ---- end to end from pinned host buffers: HostStepPipeline, one
    # dsa_decode_fused layer per step with the step's inputs (one packed
    # block) copied in and its output copied out on side streams, so that
    # the copies of one step overlap the layers of its neighbours.  The
    # steps cycle through the input copies' caches (no L2 reuse), and one
    # event pair brackets all KE steps, copies included.
    e2e = None
    if not args.no_e2e:
        B, nq, mp = spec.batch, spec.q_per_req, wl.max_pages
        pipe = api.HostStepPipeline(B, nq, H, k, mp, wl.num_pages, max_seqlen, spec.sm_scale,
                                    splits, device=dev)
        lay = pipe.layout
        host_in = [torch.zeros(lay.bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
        for hb in host_in:
            hv = api.step_views(hb, lay, B, nq, H, mp)
            for n in ("q_fp8", "q_scale", "w", "q", "seqlens", "page_table"):
                hv[n].copy_(getattr(wl, n).cpu())
        host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = int(lay.bytes)
        d2h = host_out[0].numel() * host_out[0].element_size()
        KE = max(1, min(K, 500))

        def e2e_step(i):
            c = copies[i % len(copies)]
            pipe.submit(host_in[i % 2], host_out[i % 2], c.k_fp8, c.k_scale, c.kv, stream=stream)

        for i in range(4):
            e2e_step(i)
        pipe.drain(stream)
        torch.cuda.synchronize()
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        dist_barrier(world)
        torch.cuda.synchronize()
        e_start.record(stream)
        for i in range(KE):
            e2e_step(i)
        pipe.drain(stream)
        e_end.record(stream)
        torch.cuda.synchronize()
        e2e_ms = dist_max(e_start.elapsed_time(e_end), world)
        e2e = {"value": throughput(units["query_tokens"], KE, world, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / KE,
               "note": "HostStepPipeline: per step the inputs (index/MLA queries, weights, "
                       "scales, seqlens, page table) in one pinned host block copied in, one "
                       "dsa_decode_fused layer, the output copied back to pinned host memory; "
                       "copies on side streams overlap the neighbouring steps' layers; one "
                       "event pair around all steps; the KV caches stay resident in HBM as "
                       "model state (the steps cycle through the input copies' caches)"}
        if not torch.allclose(host_out[(KE - 1) % 2], out.cpu()):
            raise RuntimeError("e2e output differs from the device output")
    del copies

    # ---- CPU oracle baseline (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, spent, nreq = OracleSampler(wl).sample(args.cpu_seconds)
        rps = n / spent
        cpu = {"value": rps, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n} query rows ({nreq} whole requests of {args.workload}, one at a time, "
                         f"cycling over its {spec.batch} requests, {spent:.1f} s of oracle time), "
                         "float64 numpy oracle (BLAS threads = cores)"}
        # the same oracle with every thread pinned to one core
        with OneCore() as one:
            if one.ok:
                n1, spent1, nreq1 = OracleSampler(wl).sample(args.cpu_seconds / 2)
                cpu["one_core"] = {"value": n1 / spent1, "unit": UNIT, "cores": 1,
                                   "sample": f"{n1} query rows ({nreq1} whole requests), "
                                             f"{spent1:.1f} s of oracle time, every thread of "
                                             "the process pinned to one core"}

    configs = None
    if rank == 0 and not args.no_configs:
        configs = measure_configs(torch, api, W, dev, K)

    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    idx_mean_ms = statistics.mean(idx_ms)
    idx_gbs = units["indexer_bytes"] / (idx_mean_ms / 1e3) / 1e9
    layer_gbs = units["layer_bytes"] / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 (indexer) + bf16 (MLA), fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": spec.batch, "q_per_req": spec.q_per_req,
                   "seqlen": spec.seqlen, "topk": k, "heads": H, "index_heads": 64,
                   "page_size": 64, "num_splits": splits,
                   "l2": (f"not flushed: the steps cycle through {args.copies} copies of the "
                          "inputs (each layer its own caches and queries), so a step's inputs "
                          f"were last touched {args.copies} layers earlier"),
                   "timed_region": f"{K} dsa_decode_fused calls (workspace clear + indexer + "
                                   "top-k + sparse MLA + merge each) back to back, "
                                   + timed_how + "; one event pair around all of them",
                   "parallelism": f"replicas x{world} (independent batches per GPU)"},
        "us_per_layer": ms_per_step * 1e3,
        "us_per_layer_single_graph_flushed": {
            "median": statistics.median(step_ms) * 1e3, "p10": pctl(step_ms, 0.1) * 1e3,
            "p90": pctl(step_ms, 0.9) * 1e3,
            "note": f"{KP} steps, each one layer per graph replay with L2 flushed before it "
                    "(flush outside the events): includes each replay's launch latency"
                    + ("" if graph is not None else "; graph capture failed: "
                       + "; ".join(capture_errors))},
        "layer_bytes": units["layer_bytes"],
        "layer_gbs": layer_gbs,
        "layer_frac_of_8tbs": layer_gbs / TARGET_HBM_GBS,
        "layer_frac_of_measured_hbm": layer_gbs / hbm,
        "stage_us": {"indexer": idx_mean_ms * 1e3, "topk": statistics.mean(topk_ms) * 1e3,
                     "sparse_mla": statistics.mean(mla_ms) * 1e3,
                     "merge": statistics.mean(merge_ms) * 1e3,
                     "note": f"separate pass of {KS} steps, an event before each kernel"},
        "roofline": {"kernel": "indexer_kernel", "bound": "hbm", "achieved": idx_gbs, "peak": hbm,
                     "unit": "GB/s", "frac": idx_gbs / hbm,
                     "traffic": indexer_traffic(args.workload),
                     "algorithmic_bytes": units["indexer_bytes"],
                     "peak_kind": f"{peak_kind} HBM copy (MEASURED_PEAKS.json hbm_gbs)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * (4 + (1 if splits > 1 else 0)),
        "clocks": clocks,
        "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
