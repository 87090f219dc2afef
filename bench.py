"""Benchmark of one TwoTower denoiser step on B300: two-segment attention + confidence unmasking.

A step is one pass of the whole hot path over one batch: attention of the S=16 block
queries of every sequence against its paged context KV and its own block KV (one
layer), followed by the unmasking of the block over the V=131072 logits.  The default
workload is the 8K-context batch: B=32 sequences of 8192 context tokens each, 64-token
pages in shuffled order, 32 query / 2 KV heads, head_dim 128, bf16.  All inputs are
seeded synthetic tensors resident in HBM before timing starts; two copies of the KV
pools and logits alternate between steps, so nothing a step reads is left in L2 by the
step before it (one copy of a step's inputs, 405 MB, is already over 3x the L2).

Prints one JSON line.  ``--impl reference`` times the float64 CPU oracle instead, on a
bounded sample of the same workload.  Under torchrun each rank runs its own batch
(sequences are independent: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_wise_diffusion_denoise_b300 import synth  # noqa: E402

WORKLOADS = {
    "ctx8k": "ctx8k", "single": "single", "ragged": "ragged", "long": "long", "loop": "loop",
}


def parse():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(WORKLOADS), default="ctx8k")
    ap.add_argument("--no-graph", action="store_true", help="launch every step from Python")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--s-variants", dest="s_variants", action="store_true", default=True,
                    help="also time the attention at block sizes S = 32, 64, 128 on the same contexts (default)")
    ap.add_argument("--no-s-variants", dest="s_variants", action="store_false",
                    help="skip the block-size timings")
    ap.add_argument("--loop-blocks", type=int, default=0,
                    help="(--config loop) blocks per loop instead of the workload's 8 (a smaller run to profile)")
    ap.add_argument("--loop-steps", type=int, default=0,
                    help="(--config loop) denoise steps per block instead of the workload's T = 16")
    ap.add_argument("--tau", type=float, default=None,
                    help="confidence threshold instead of the workload's 0.9 (e.g. 0.8, the other operating point)")
    return ap.parse_args()


# --------------------------------------------------------------------------- algorithmic cost

CSRC = os.path.join(ROOT, "block_wise_diffusion_denoise_b300", "csrc")
PROFILED = {   # kernel -> (summary under profiles/, the sources its counters were taken from)
    "attention": ("attention_ctx8k.md", ("attn_tc.cu", "attn_work.cuh", "sm100_ptx.cuh", "tt_common.cuh")),
    "unmask": ("unmask_ctx8k.md", ("unmask.cu", "vocab_stream.cuh", "sm100_ptx.cuh", "tt_common.cuh")),
    "masked_nll": ("masked_nll_ctx8k.md", ("masked_nll.cu", "vocab_stream.cuh", "sm100_ptx.cuh", "tt_common.cuh")),
    "decode": ("decode_attention_ctx8k.md", ("attn_decode.cu", "attn_work.cuh", "sm100_ptx.cuh", "tt_common.cuh")),
}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary, or None when the
    summary is for another workload or the kernel's sources have changed since the capture."""
    import hashlib
    name, files = PROFILED[kernel]
    path = os.path.join(ROOT, "profiles", name)
    if workload != "ctx8k" or not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.split(":", 1)[0] in ("kernel_sources_sha256", "traffic_bytes_per_launch"):
            k, v = line.split(":", 1)
            fields[k] = v.split()[0]
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    if fields.get("kernel_sources_sha256") != h.hexdigest()[:16] or "traffic_bytes_per_launch" not in fields:
        return None
    return int(fields["traffic_bytes_per_launch"])


def attn_bytes(cfg, lens) -> float:
    """Bytes a perfect attention kernel moves: context K/V once, q, block K/V and the output."""
    elem = 2 if cfg.dtype == "bf16" else 4
    per_seq_fixed = (cfg.S * cfg.Hq * cfg.D * 2 + cfg.S * cfg.Hkv * cfg.D * 2) * elem
    return float(sum(2 * int(L) * cfg.Hkv * cfg.D * elem for L in lens) + cfg.B * per_seq_fixed)


def attn_flops(cfg, lens) -> float:
    return float(sum(4.0 * cfg.Hq * cfg.S * cfg.D * (int(L) + cfg.S) for L in lens))


def s_var_entry(cfg, lens, Sv, us, hbm, tc):
    """Timing of the attention at block size Sv against its own roofline (bytes grow a little with
    S, flops in proportion: from S = 32 on the tensor bound takes over)."""
    c2 = cfg.replace(S=Sv)
    ab, af = attn_bytes(c2, lens), attn_flops(c2, lens)
    t_hbm, t_tc = ab / (hbm * 1e9), af / (tc * 1e12)
    roof = max(t_hbm, t_tc) * 1e6
    return {"us": us, "roofline_us": roof, "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": roof / us,
            "gbs": ab / (us * 1e-6) / 1e9, "tflops": af / (us * 1e-6) / 1e12}


def unmask_bytes(cfg, masked_rows) -> float:
    elem = 2 if cfg.dtype == "bf16" else 4
    return float(masked_rows * cfg.V * elem)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples the SM clock and throttle reasons while the timed region runs: NVML from a
    thread when the Python bindings are present, otherwise an ``nvidia-smi -lms`` child."""
    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        import torch
        self.samples, self.reasons, self.mode, self.max_mhz = [], set(), None, None
        self._stop = threading.Event()
        pr = torch.cuda.get_device_properties(index)
        self.bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            try:
                self.h = pynvml.nvmlDeviceGetHandleByPciBusId(self.bus)
            except Exception:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception:
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "smi"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                r = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for name, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(0.002)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        elif self.mode == "smi":
            import subprocess
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.bus, f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)          # let the first sample land before the timed region
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self.t.join()
        elif self.mode == "smi":
            time.sleep(0.05)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6 or not f[0].isdigit():
                    continue
                self.samples.append(int(f[0]))
                self.max_mhz = int(f[1]) if f[1].isdigit() else self.max_mhz
                for name, val in zip(names, f[2:6]):
                    if val.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        if self.mode is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": "no NVML and no nvidia-smi"}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": self.mode}


# --------------------------------------------------------------------------- CPU oracle timing

class OracleSampler:
    """Times the float64 oracle on a bounded sample of the workload: (sequence, KV head)
    attention pairs and single unmask rows, scaled to one full batch step."""

    def __init__(self, cfg, seed):
        import oracle
        self.oracle, self.cfg = oracle, cfg
        self.lens = synth.draw_lengths(cfg, seed)
        self.cache = synth.draw_paged_cache(cfg, self.lens, int(self.lens.max()) + cfg.S, seed=seed)
        self.q, self.kb, self.vb = synth.draw_block_qkv(cfg, seed=seed)
        self.lg = synth.draw_logits(cfg, seed=seed, rows=1)
        self.n_pairs = self.n_rows = 0
        self.t_attn = self.t_unm = 0.0

    def one(self):
        """One attention pair and one unmask row; returns their seconds."""
        cfg, o, c = self.cfg, self.oracle, self.cache
        b = (self.n_pairs // cfg.Hkv) % cfg.B
        g = self.n_pairs % cfg.Hkv
        L = int(self.lens[b])
        t0 = time.perf_counter()
        kc = o.decode(o.context_rows(c.k_pool, c.page_table[b], L, cfg.page_size), cfg.dtype)
        vc = o.decode(o.context_rows(c.v_pool, c.page_table[b], L, cfg.page_size), cfg.dtype)
        hs = slice(g * cfg.G, (g + 1) * cfg.G)
        o.denoise_attention_seq(o.decode(self.q[b][:, hs], cfg.dtype), kc[:, g:g + 1], vc[:, g:g + 1],
                                o.decode(self.kb[b][:, g:g + 1], cfg.dtype),
                                o.decode(self.vb[b][:, g:g + 1], cfg.dtype), 1.0 / math.sqrt(cfg.D))
        t1 = time.perf_counter()
        masked = np.zeros((1, cfg.S), np.uint8)
        masked[0, self.n_rows % cfg.S] = 1
        o.unmask(self.lg, masked, np.full((1, cfg.S), -1), cfg.tau, 1, cfg.T, cfg.dtype)
        t2 = time.perf_counter()
        self.n_pairs += 1
        self.n_rows += 1
        self.t_attn += t1 - t0
        self.t_unm += t2 - t1
        return t1 - t0, t2 - t1

    def scale(self, t_pair, t_row):
        """Seconds of one full batch step from the time of one pair and one row."""
        return t_pair * self.cfg.B * self.cfg.Hkv + t_row * self.cfg.B * self.cfg.S

    def run(self, budget_s):
        t_end = time.perf_counter() + budget_s
        while time.perf_counter() < t_end or self.n_pairs == 0:
            self.one()
        per_step = self.scale(self.t_attn / self.n_pairs, self.t_unm / self.n_rows)
        return per_step, self.t_attn + self.t_unm

    def note(self):
        cfg = self.cfg
        return (f"{self.n_pairs} (sequence, KV head) attention pairs and {self.n_rows} unmask rows of the "
                f"{cfg.name} workload, scaled to the full batch of {cfg.B} x {cfg.Hkv} pairs and "
                f"{cfg.B * cfg.S} rows")


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        th = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        th = os.cpu_count()
    return int(th)


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_reference(a, cfg):
    """The oracle arm.  A step here is a bounded sample of one batch step -- one
    (sequence, KV head) attention pair and one unmask row, timed on the host cores --
    so that K steps take seconds, not the ~3 s each a whole batch step takes.  The
    line's ms_per_step is that sample's measured time (what the run spent per step);
    value is the full batch's steps/s, the sample's time scaled by its share of the
    batch (sample_fraction)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    smp = OracleSampler(cfg, a.seed)
    for _ in range(a.warmup):
        smp.one()
    t0 = time.perf_counter()
    samples = [smp.one() for _ in range(a.steps)]
    wall = time.perf_counter() - t0
    t_pair = sum(x[0] for x in samples) / len(samples)
    t_row = sum(x[1] for x in samples) / len(samples)
    full_step = smp.scale(t_pair, t_row)               # seconds of one whole batch step
    sample_step = t_pair + t_row                       # seconds of one sampled step
    value = 1.0 / full_step
    note = (f"per step, one (sequence, KV head) attention pair and one unmask row of the {cfg.name} "
            f"workload (measured: {sample_step * 1e3:.1f} ms per step); value scales them to "
            f"{cfg.B} x {cfg.Hkv} pairs and {cfg.B * cfg.S} rows ({full_step:.2f} s per batch step)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": sample_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg, a), "wall_s": wall,
            "sample_fraction": sample_step / full_step, "full_step_ms": full_step * 1e3,
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cpu_cores(), "cpu": cpu_model(),
                             "kind": "oracle", "sample": note},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


METRIC = "denoise steps/s (attn+unmask) at ctx 8K, S=16; % of HBM/tensor roofline"


def config_dict(cfg, a):
    return {"workload": f"{cfg.name}: B={cfg.B}, context {cfg.len_lo}"
                        + (f"-{cfg.len_hi}" if cfg.len_hi != cfg.len_lo else "")
                        + f", S={cfg.S}, {cfg.Hq}q/{cfg.Hkv}kv heads, head_dim {cfg.D}, vocab {cfg.V}, "
                          f"{cfg.page_size}-token shuffled pages, tau={cfg.tau}, one attention layer + unmask per step",
            "global_batch": cfg.B * a.gpus, "seq_len": cfg.len_hi, "block": cfg.S,
            "parallelism": f"dp{a.gpus} (independent sequences)",
            "l2": "inputs larger than L2, two copies alternate between steps"}


# --------------------------------------------------------------------------- ranks

def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of its own batch in at most max_ms."""
    return world * steps / (max_ms / 1e3)


# --------------------------------------------------------------------------- GPU arm

def run_ours(a, cfg):
    import torch
    import torch.distributed as dist

    from block_wise_diffusion_denoise_b300 import api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    # ---- inputs, resident in HBM; rank r draws its own batch (independent sequences)
    seed = a.seed + 1000 * rank
    lens = synth.draw_lengths(cfg, seed)
    cap = int(lens.max()) + cfg.S
    cache_h = synth.draw_paged_cache(cfg, lens, cap, seed=seed)
    q_h, kb_h, vb_h = synth.draw_block_qkv(cfg, seed=seed)
    lg_h = synth.draw_logits(cfg, seed=seed)

    def dev_t(x):
        if cfg.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    n_copies = 2
    base = {"k": dev_t(cache_h.k_pool), "v": dev_t(cache_h.v_pool), "lg": dev_t(lg_h)}
    table = torch.from_numpy(cache_h.page_table).to(dev)
    ctx_len = torch.from_numpy(cache_h.ctx_len).to(dev)
    copies = []
    for c in range(n_copies):
        k = base["k"] if c == 0 else base["k"].clone()
        v = base["v"] if c == 0 else base["v"].clone()
        lg = base["lg"] if c == 0 else base["lg"].clone()
        copies.append({"cache": api.KVCache(k, v, table, ctx_len), "q": dev_t(q_h), "kb": dev_t(kb_h),
                       "vb": dev_t(vb_h), "lg": lg, "out": torch.empty(q_h.shape, dtype=base["k"].dtype,
                                                                        device=dev)})
    tdt = base["k"].dtype
    ws = api.workspace(api.tt_block_step_workspace_size(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.D, cfg.V, tdt), dev)
    attn_ws = api.workspace(api.tt_denoise_attn_workspace_size(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.D, tdt), dev)
    unm_ws = api.workspace(api.tt_unmask_workspace_size(cfg.B, cfg.S, cfg.V, tdt), dev)
    err = api.error_word(dev)
    n_state = a.warmup + a.steps
    # every step starts a fresh block (all 16 positions masked, step 1): fresh state per step
    masked = torch.ones((n_state, cfg.B, cfg.S), dtype=torch.uint8, device=dev)
    tokens = torch.full((n_state, cfg.B, cfg.S), -1, dtype=torch.int32, device=dev)
    committed = torch.zeros((n_state, cfg.B, cfg.S), dtype=torch.uint8, device=dev)
    n_masked = torch.zeros((n_state, cfg.B), dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(cfg.D)

    def step(i, stream=None):
        c = copies[i % n_copies]
        api.tt_block_step([c["cache"]], [c["q"]], [c["kb"]], [c["vb"]], [c["out"]], c["lg"], masked[i],
                          tokens[i], cfg.tau, 1, cfg.T, sm_scale=scale, committed_now=committed[i],
                          n_masked=n_masked[i], ws=ws, dev_err=err, stream=stream)

    def attn_only(i, stream=None):
        c = copies[i % n_copies]
        api.tt_denoise_attn(c["cache"], c["q"], c["kb"], c["vb"], out=c["out"], sm_scale=scale, ws=attn_ws,
                            dev_err=err, stream=stream)

    def ctx_attn_only(i, stream=None):
        c = copies[i % n_copies]
        api.tt_context_block_attn(c["cache"], c["q"], c["kb"], c["vb"], out=c["out"], sm_scale=scale,
                                  ws=attn_ws, dev_err=err, stream=stream)

    k_ker = max(10, min(a.steps, 200))   # launches per kernel-only timing
    unm_masked = torch.ones((k_ker, cfg.B, cfg.S), dtype=torch.uint8, device=dev)
    unm_tokens = torch.full((k_ker, cfg.B, cfg.S), -1, dtype=torch.int32, device=dev)

    def unmask_only(i, stream=None):
        c = copies[i % n_copies]
        api.tt_unmask(c["lg"], unm_masked[i], unm_tokens[i], cfg.tau, 1, cfg.T, ws=unm_ws, dev_err=err,
                      stream=stream)

    # the masked-diffusion loss over the same logits, every position masked (the unmasking's
    # bytes: masked rows x V)
    nll_ws = api.workspace(api.tt_masked_nll_workspace_size(cfg.B, cfg.S, cfg.V, tdt), dev)
    nll_targets = torch.from_numpy(synth.draw_corruption(cfg, seed)[0]).to(dev)
    nll_masked = torch.ones((cfg.B, cfg.S), dtype=torch.uint8, device=dev)
    nll_out = torch.empty((cfg.B, cfg.S), dtype=torch.float32, device=dev)
    nll_sum = torch.empty((cfg.B,), dtype=torch.float32, device=dev)
    nll_cnt = torch.empty((cfg.B,), dtype=torch.int32, device=dev)

    def nll_only(i, stream=None):
        c = copies[i % n_copies]
        api.tt_masked_nll(c["lg"], nll_targets, nll_masked, nll=nll_out, nll_sum=nll_sum, count=nll_cnt, ws=nll_ws,
                          dev_err=err, stream=stream)

    # one decoding position (S = 1) per sequence on the same caches: the first block position's
    # q / k / v (the decode kernel; every query head of a KV head in one pass over the context)
    dec = [{"q": c["q"][:, :1].contiguous(), "kb": c["kb"][:, :1].contiguous(), "vb": c["vb"][:, :1].contiguous(),
            "out": torch.empty_like(c["q"][:, :1])} for c in copies]
    dec_ws = api.workspace(api.tt_denoise_attn_workspace_size(cfg.B, 1, cfg.Hq, cfg.Hkv, cfg.D, tdt), dev)

    def decode_only(i, stream=None):
        c, d = copies[i % n_copies], dec[i % n_copies]
        api.tt_denoise_attn(c["cache"], d["q"], d["kb"], d["vb"], out=d["out"], sm_scale=scale, ws=dec_ws,
                            dev_err=err, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def timed(fn, first, count, use_graph):
        """Run fn(first .. first+count-1) and return (ms total) by CUDA events on the launching stream."""
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        if use_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(first, first + count):
                    fn(i, stream=s)
            barrier()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                ev0.record(s)
                g.replay()
                ev1.record(s)
        else:
            barrier()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(s)
            for i in range(first, first + count):
                fn(i, stream=s)
            ev1.record(s)
        ev1.synchronize()
        return ev0.elapsed_time(ev1)

    use_graph = not a.no_graph
    # ---- warm-up (eager), then the timed region: exactly K steps
    for i in range(a.warmup):
        step(i)
    barrier()
    masked[a.warmup:].fill_(1)
    sampler = ClockSampler(local)
    if use_graph:
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(a.warmup, a.warmup + a.steps):
                step(i, stream=s)
        masked[a.warmup:].fill_(1)
        tokens[a.warmup:].fill_(-1)
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with sampler, torch.cuda.stream(s):
            ev0.record(s)
            g.replay()
            ev1.record(s)
            ev1.synchronize()
    else:
        s = torch.cuda.current_stream()
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with sampler:
            ev0.record(s)
            for i in range(a.warmup, a.warmup + a.steps):
                step(i)
            ev1.record(s)
            ev1.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world, dev)
    code = api.tt_get_device_error(err)
    if code != 0:
        raise SystemExit(f"device error {code} during the timed region")
    # the timed steps really unmasked: every sequence committed at least one position
    if int(committed[a.warmup:].sum(dim=2).min().item()) < 1:
        raise SystemExit("a timed step committed nothing")

    # ---- per-kernel durations (CUDA events on the launching stream), same rotation of inputs
    attn_ms = timed(attn_only, 0, k_ker, use_graph) / k_ker
    unm_masked.fill_(1)
    unmask_ms = timed(unmask_only, 0, k_ker, use_graph) / k_ker
    # the context tower's causal view of the same block (not part of the denoise step)
    ctx_attn_ms = timed(ctx_attn_only, 0, k_ker, use_graph) / k_ker
    # the training-side loss over the same logits (not part of the denoise step)
    nll_ms = timed(nll_only, 0, k_ker, use_graph) / k_ker
    # one autoregressive decoding step's attention on the same contexts (S = 1)
    dec_ms = timed(decode_only, 0, k_ker, use_graph) / k_ker
    # positions the timed denoise steps committed (the first step of a fresh block)
    commits = float(committed[a.warmup:].sum().item()) / a.steps
    # block sizes S = 32, 64, 128 on the same contexts (the attention alone)
    s_var = {}
    if a.s_variants:
        for Sv in (32, 64, 128):
            g = torch.Generator(device=dev)
            g.manual_seed(Sv)
            qv = (torch.randn((cfg.B, Sv, cfg.Hq, cfg.D), generator=g, device=dev) * scale).to(tdt)
            kv_ = (torch.randn((cfg.B, Sv, cfg.Hkv, cfg.D), generator=g, device=dev) * scale).to(tdt)
            vv_ = (torch.randn((cfg.B, Sv, cfg.Hkv, cfg.D), generator=g, device=dev) * scale).to(tdt)
            ov = torch.empty_like(qv)
            wsv = api.workspace(api.tt_denoise_attn_workspace_size(cfg.B, Sv, cfg.Hq, cfg.Hkv, cfg.D, tdt), dev)

            def attn_sv(i, stream=None, qv=qv, kv_=kv_, vv_=vv_, ov=ov, wsv=wsv):
                c = copies[i % n_copies]
                api.tt_denoise_attn(c["cache"], qv, kv_, vv_, out=ov, sm_scale=scale, ws=wsv, dev_err=err,
                                    stream=stream)
            s_var[Sv] = timed(attn_sv, 0, k_ker, use_graph) / k_ker
    if api.tt_get_device_error(err) != 0:
        raise SystemExit("device error in the per-kernel timings")

    # ---- end to end through the public API with host buffers (pinned), copies inside the region
    e2e = None
    if a.e2e_steps > 0:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        c0 = copies[0]
        h_q, h_kb, h_vb, h_lg = pin(c0["q"]), pin(c0["kb"]), pin(c0["vb"]), pin(c0["lg"])
        h_out = torch.empty(c0["out"].shape, dtype=c0["out"].dtype).pin_memory()
        h_tok = torch.empty((cfg.B, cfg.S), dtype=torch.int32).pin_memory()
        h_msk = torch.empty((cfg.B, cfg.S), dtype=torch.uint8).pin_memory()
        h_msk_in = torch.ones((cfg.B, cfg.S), dtype=torch.uint8).pin_memory()
        h_tok_in = torch.full((cfg.B, cfg.S), -1, dtype=torch.int32).pin_memory()
        d = {k: torch.empty_like(v, device=dev) for k, v in
             (("q", h_q), ("kb", h_kb), ("vb", h_vb), ("lg", h_lg))}
        d_m = torch.empty((cfg.B, cfg.S), dtype=torch.uint8, device=dev)
        d_t = torch.empty((cfg.B, cfg.S), dtype=torch.int32, device=dev)
        d_o = torch.empty_like(c0["out"])
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kb, h_vb, h_lg, h_msk_in, h_tok_in))
        d2h = sum(t.numel() * t.element_size() for t in (h_out, h_tok, h_msk))

        # The logits (almost all of a step's input bytes) cross the host link in four
        # chunks on side streams, which moves about 15 % more per second than one copy.
        side = [torch.cuda.Stream(device=dev) for _ in range(4)]
        lg_h_flat, lg_d_flat = h_lg.view(-1), d["lg"].view(-1)
        chunk = (lg_h_flat.numel() + len(side) - 1) // len(side)

        def e2e_step():
            main = torch.cuda.current_stream()
            for k, h in (("q", h_q), ("kb", h_kb), ("vb", h_vb)):
                d[k].copy_(h, non_blocking=True)
            for i, s in enumerate(side):
                s.wait_stream(main)            # the previous step has finished reading them
                with torch.cuda.stream(s):
                    lg_d_flat[i * chunk:(i + 1) * chunk].copy_(lg_h_flat[i * chunk:(i + 1) * chunk],
                                                               non_blocking=True)
            for s in side:
                main.wait_stream(s)
            d_m.copy_(h_msk_in, non_blocking=True)
            d_t.copy_(h_tok_in, non_blocking=True)
            api.tt_block_step([c0["cache"]], [d["q"]], [d["kb"]], [d["vb"]], [d_o], d["lg"], d_m, d_t, cfg.tau,
                              1, cfg.T, sm_scale=scale, ws=ws, dev_err=err)
            h_out.copy_(d_o, non_blocking=True)
            h_tok.copy_(d_t, non_blocking=True)
            h_msk.copy_(d_m, non_blocking=True)

        for _ in range(2):
            e2e_step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(a.e2e_steps):
            e2e_step()
        e1.record()
        e1.synchronize()
        e_ms = e0.elapsed_time(e1) / a.e2e_steps
        e_ms = max_over_ranks(e_ms, world, dev)
        e2e = {"value": job_rate(world, 1, e_ms), "unit": "steps/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": a.e2e_steps,
               "link_gbs": (h2d + d2h) / (e_ms * 1e-3) / 1e9,
               "note": "bound by the host link: the step's logits cross it every step; link_gbs = bytes "
                       "moved per step / the step's time"}

    if rank == 0:
        import json as _json
        peaks = _json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
            if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
        hbm = peaks.get("hbm_gbs", 6400.0)
        tc = peaks.get("bf16_tflops", 1800.0)
        src = "of measured" if peaks else "of fallback"
        ab, af = attn_bytes(cfg, lens), attn_flops(cfg, lens)
        ub = unmask_bytes(cfg, cfg.B * cfg.S)
        db = attn_bytes(cfg.replace(S=1), lens)
        attn_gbs = ab / (attn_ms * 1e-3) / 1e9
        attn_tfs = af / (attn_ms * 1e-3) / 1e12
        unm_gbs = ub / (unmask_ms * 1e-3) / 1e9
        step_roof_us = max(ab / (hbm * 1e9), af / (tc * 1e12)) * 1e6 + ub / (hbm * 1e9) * 1e6
        value = job_rate(world, a.steps, ms)
        line = {
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded; value distributions of the "
                                                              "workload recipe)",
            "config": config_dict(cfg, a),
            "roofline": {"bound": "hbm", "kernel": "denoise attention", "achieved": attn_gbs, "peak": hbm,
                         "unit": "GB/s", "frac": attn_gbs / hbm, "peak_source": src,
                         "algorithmic_bytes_per_launch": ab, "avg_launch_us": attn_ms * 1e3,
                         "tensor_tflops": attn_tfs, "tensor_frac": attn_tfs / tc,
                         "traffic": profiled_traffic("attention", cfg.name),
                         "traffic_source": "profiles/attention_ctx8k.md (ncu dram__bytes_read.sum + "
                                           "dram__bytes_write.sum, one launch)"},
            "kernels": {
                "attention": {"us": attn_ms * 1e3, "gbs": attn_gbs, "hbm_frac": attn_gbs / hbm,
                              "roofline_us": max(ab / (hbm * 1e9), af / (tc * 1e12)) * 1e6},
                "unmask": {"us": unmask_ms * 1e3, "gbs": unm_gbs, "hbm_frac": unm_gbs / hbm,
                           "roofline_us": ub / (hbm * 1e9) * 1e6,
                           "traffic": profiled_traffic("unmask", cfg.name)},
                "context_block_attention": {
                    "us": ctx_attn_ms * 1e3, "gbs": ab / (ctx_attn_ms * 1e-3) / 1e9,
                    "hbm_frac": ab / (ctx_attn_ms * 1e-3) / 1e9 / hbm,
                    "roofline_us": max(ab / (hbm * 1e9), af / (tc * 1e12)) * 1e6,
                    "note": "tt_context_block_attn on the same inputs; timed separately, not in the step"},
                "masked_nll": {
                    "us": nll_ms * 1e3, "gbs": ub / (nll_ms * 1e-3) / 1e9, "hbm_frac": ub / (nll_ms * 1e-3) / 1e9 / hbm,
                    "roofline_us": ub / (hbm * 1e9) * 1e6, "traffic": profiled_traffic("masked_nll", cfg.name),
                    "note": "tt_masked_nll over the step's logits with every position masked; timed separately, "
                            "not in the step"},
                "decode_attention": {
                    "us": dec_ms * 1e3, "gbs": db / (dec_ms * 1e-3) / 1e9, "hbm_frac": db / (dec_ms * 1e-3) / 1e9 / hbm,
                    "roofline_us": db / (hbm * 1e9) * 1e6, "traffic": profiled_traffic("decode", cfg.name),
                    "note": "one position per sequence (S = 1, the AR decoding step) on the same caches: "
                            "tt_denoise_attn's decode kernel; timed separately, not in the step"},
                "step_roofline_us": step_roof_us, "step_frac": step_roof_us / (ms / a.steps * 1e3)},
            "attention_per_committed_token": {
                "unit": "us of attention per committed token (all sequences of the batch)",
                "block_diffusion": attn_ms * 1e3 / commits, "ar_decode": dec_ms * 1e3 / cfg.B,
                "ratio_ar_over_diffusion": (dec_ms / cfg.B) / (attn_ms / commits),
                "commits_per_step": commits,
                "note": "diffusion: the S=16 block attention per step / positions the timed steps committed "
                        "(first denoise step of a fresh block on the synthetic logits); AR: the S=1 attention "
                        "per step / B (one token per sequence). Per layer; the model's other layers are out "
                        "of scope"},
            "attention_block_sizes": {
                f"S{Sv}": s_var_entry(cfg, lens, Sv, us * 1e3, hbm, tc) for Sv, us in s_var.items()},
            "gpu_launches": a.steps * launches_per_step(cfg),
            "graph": use_graph,
            "clocks": sampler.summary(),
        }
        if e2e is not None:
            line["e2e"] = e2e
        if not a.no_cpu_baseline:
            smp = OracleSampler(cfg, a.seed)
            per_step, spent = smp.run(12.0)
            line["cpu_baseline"] = {"value": 1.0 / per_step, "unit": "steps/s", "cores": cpu_cores(),
                                    "cpu": cpu_model(), "kind": "oracle",
                                    "sample": smp.note() + f" ({spent:.1f} s of CPU time)"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------- the block loop

def run_loop(a, cfg):
    """The full block loop: B sequences with their own paged caches in every one of n_layers
    attention layers, n_blocks consecutive blocks of S positions, each refined for T steps
    (tt_block_step: every layer's attention, then the unmasking of the step's logits) and then
    committed into every layer's cache (tt_kv_append), all replayed from one CUDA graph.

    Values: pools and block q/k/v ~ N(0,1)/sqrt(D), step logits ~ N(0,3) plus a peak U[0,12]
    at a uniform token per position, committed-block K/V ~ N(0,1), all drawn on the device
    from torch generators seeded by (seed, block, step, layer); page tables from synth."""
    import torch
    import torch.distributed as dist

    from block_wise_diffusion_denoise_b300 import api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    bf = torch.bfloat16
    seed = a.seed + 1000 * rank
    if a.loop_blocks > 0 or a.loop_steps > 0:
        cfg = cfg.replace(n_blocks=a.loop_blocks or cfg.n_blocks, T=a.loop_steps or cfg.T)
    B, S, Hq, Hkv, D, V, T, NL, NB = cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.D, cfg.V, cfg.T, cfg.n_layers, cfg.n_blocks
    L0 = cfg.len_lo
    cap = L0 + S * NB
    table_h, num_pages = synth.draw_page_table(cfg, cap, seed)
    table = torch.from_numpy(table_h).to(dev)
    ctx0 = torch.full((B,), L0, dtype=torch.int32, device=dev)
    ctx_len = ctx0.clone()

    import zlib

    def gen(*key):
        g = torch.Generator(device=dev)
        g.manual_seed(zlib.crc32(repr((seed,) + key).encode()))
        return g

    def normal(shape, scale, key):
        return (torch.randn(shape, generator=gen(*key), device=dev, dtype=torch.float32) * scale).to(bf)

    sc = 1.0 / math.sqrt(D)
    caches = [api.KVCache(normal((num_pages, Hkv, cfg.page_size, D), sc, ("k", l)),
                          normal((num_pages, Hkv, cfg.page_size, D), sc, ("v", l)), table, ctx_len)
              for l in range(NL)]
    # block q/k/v: two rotating sets per layer (their values do not change the work)
    qkv = [[(normal((B, S, Hq, D), sc, ("q", l, r)), normal((B, S, Hkv, D), sc, ("kb", l, r)),
             normal((B, S, Hkv, D), sc, ("vb", l, r))) for l in range(NL)] for r in range(2)]
    outs = [torch.empty((B, S, Hq, D), dtype=bf, device=dev) for _ in range(NL)]
    logits = []
    for blk in range(NB):
        for st in range(T):
            g = gen("lg", blk, st)
            x = torch.randn((B, S, V), generator=g, device=dev, dtype=torch.float32) * cfg.logit_std
            tok = torch.randint(0, V, (B, S), generator=g, device=dev)
            h = torch.rand((B, S), generator=g, device=dev) * cfg.peak_hi
            x.view(B * S, V)[torch.arange(B * S, device=dev), tok.view(-1)] += h.view(-1)
            logits.append(x.to(bf))
            del x
    knew = [[normal((B, S, Hkv, D), 1.0, ("kn", blk, l)) for l in range(NL)] for blk in range(NB)]
    vnew = [[normal((B, S, Hkv, D), 1.0, ("vn", blk, l)) for l in range(NL)] for blk in range(NB)]
    masked = torch.ones((B, S), dtype=torch.uint8, device=dev)
    tokens = torch.full((B, S), -1, dtype=torch.int32, device=dev)
    nsteps = NB * T
    com = torch.zeros((nsteps, B, S), dtype=torch.uint8, device=dev)
    nm = torch.zeros((nsteps, B), dtype=torch.int32, device=dev)
    ws = api.workspace(api.tt_block_step_workspace_size(B, S, Hq, Hkv, D, V, bf), dev)
    err = api.error_word(dev)

    def loop(stream):
        ctx_len.copy_(ctx0)
        for blk in range(NB):
            masked.fill_(1)
            tokens.fill_(-1)
            for st in range(1, T + 1):
                i = blk * T + st - 1
                r = qkv[i % 2]
                api.tt_block_step(caches, [x[0] for x in r], [x[1] for x in r], [x[2] for x in r], outs, logits[i],
                                  masked, tokens, cfg.tau, st, T, sm_scale=sc, committed_now=com[i],
                                  n_masked=nm[i], ws=ws, dev_err=err, stream=stream)
            api.tt_kv_append(caches, knew[blk], vnew[blk], dev_err=err, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    s_ = torch.cuda.Stream(device=dev)
    s_.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s_):
        loop(s_)                                        # eager warm-up (and first check)
    barrier()
    if api.tt_get_device_error(err) != 0:
        raise SystemExit("device error in the block loop")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_):
        loop(s_)
    for _ in range(max(1, a.warmup)):
        g.replay()
    barrier()
    reps = max(1, a.steps // nsteps) if a.steps >= nsteps else 1
    sampler = ClockSampler(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler, torch.cuda.stream(s_):
        ev0.record(s_)
        for _ in range(reps):
            g.replay()
        ev1.record(s_)
        ev1.synchronize()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    if api.tt_get_device_error(err) != 0:
        raise SystemExit("device error in the timed block loop")
    # every block finished within T steps and every step committed at least one position
    ends = nm.view(NB, T, B)[:, T - 1]
    if int(ends.max().item()) != 0:
        raise SystemExit("a block did not finish within T steps")
    commits = com.view(NB, T, B, S).sum(dim=(2, 3)).float()    # per (block, step), whole batch
    steps_done = (commits > 0).sum().item()

    # the append alone: NB appends from the start length, timed in a graph
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga, stream=s_):
        ctx_len.copy_(ctx0)
        for blk in range(NB):
            api.tt_kv_append(caches, knew[blk], vnew[blk], dev_err=err, stream=s_)
    ga.replay()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_):
        e0.record(s_)
        for _ in range(10):
            ga.replay()
        e1.record(s_)
        e1.synchronize()
    append_us = e0.elapsed_time(e1) / (10 * NB) * 1e3

    # The attention alone, every layer at the start length: the block (S = 16) and one
    # autoregressive decoding position (S = 1) per sequence, for the attention cost per
    # committed token of the two ways of generating.
    attn_ws = api.workspace(api.tt_denoise_attn_workspace_size(B, S, Hq, Hkv, D, bf), dev)
    dec_ws = api.workspace(api.tt_denoise_attn_workspace_size(B, 1, Hq, Hkv, D, bf), dev)
    dec_qkv = [(x[0][:, :1].contiguous(), x[1][:, :1].contiguous(), x[2][:, :1].contiguous()) for x in qkv[0]]
    dec_out = [torch.empty((B, 1, Hq, D), dtype=bf, device=dev) for _ in range(NL)]

    def layers(stream, decode):
        for l in range(NL):
            if decode:
                q1, k1, v1 = dec_qkv[l]
                api.tt_denoise_attn(caches[l], q1, k1, v1, out=dec_out[l], sm_scale=sc, ws=dec_ws, dev_err=err,
                                    stream=stream)
            else:
                q, kb, vb = qkv[0][l]
                api.tt_denoise_attn(caches[l], q, kb, vb, out=outs[l], sm_scale=sc, ws=attn_ws, dev_err=err,
                                    stream=stream)

    layer_us = {}
    for decode in (False, True):
        gl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl, stream=s_):
            ctx_len.copy_(ctx0)
            for _ in range(4):
                layers(s_, decode)
        gl.replay()
        barrier()
        with torch.cuda.stream(s_):
            e0.record(s_)
            for _ in range(5):
                gl.replay()
            e1.record(s_)
            e1.synchronize()
        layer_us[decode] = e0.elapsed_time(e1) / 20 * 1e3     # all NL layers, one step
    if api.tt_get_device_error(err) != 0:
        raise SystemExit("device error in the attention-only timings")

    if rank == 0:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
            if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
        hbm = peaks.get("hbm_gbs", 6400.0)
        tc = peaks.get("bf16_tflops", 1800.0)
        # algorithmic cost of the whole loop (every layer's attention at the block's context
        # length; the unmasking reads every still-masked row; the append moves S rows per layer)
        roof_s = 0.0
        byts = 0.0
        mask_rows = nm.view(NB, T, B).sum(dim=2).cpu().numpy()
        for blk in range(NB):
            lens = np.full(B, L0 + S * blk)
            ab, af = attn_bytes(cfg, lens), attn_flops(cfg, lens)
            for st in range(T):
                masked_before = B * S if st == 0 else int(mask_rows[blk, st - 1])
                ub = unmask_bytes(cfg, masked_before)
                roof_s += NL * max(ab / (hbm * 1e9), af / (tc * 1e12)) + ub / (hbm * 1e9)
                byts += NL * ab + ub
            append_b = NL * 2 * 2 * B * S * Hkv * D * 2.0          # read + write, K and V
            roof_s += append_b / (hbm * 1e9)
            byts += append_b
        per_loop_ms = ms / reps
        value = job_rate(world, reps * nsteps, ms)
        line = {
            "metric": "block-loop denoise steps/s (6 attention layers + unmask per step, append per block)",
            "value": value, "unit": "steps/s", "n_gpus": world, "steps": reps * nsteps, "warmup": a.warmup,
            "ms_per_step": per_loop_ms / nsteps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded on the device; value distributions of the workload recipe)",
            "config": {"workload": f"loop: B={B}, initial context {L0}, S={S}, {Hq}q/{Hkv}kv heads, head_dim {D}, "
                                   f"vocab {V}, {NL} attention layers with their own paged caches, {NB} blocks of "
                                   f"T={T} steps, tau={cfg.tau}, tt_kv_append per block",
                       "l2": "inputs larger than L2 (1.6 GB of caches, 64 MB of logits per step)"},
            "roofline": {"bound": "hbm", "achieved": byts / (per_loop_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": roof_s / (per_loop_ms * 1e-3), "peak_source": "of measured" if peaks else "of fallback",
                         "roofline_ms_per_loop": roof_s * 1e3, "algorithmic_bytes_per_loop": byts},
            "commits_per_step": float(commits.sum().item() / nsteps),
            "commits_per_step_per_sequence": float(commits.sum().item() / nsteps / B),
            "steps_with_a_commit": int(steps_done),
            "kernels": {"append": {"us": append_us, "layers": NL,
                                   "bytes": NL * 2 * 2 * B * S * Hkv * D * 2.0,
                                   "gbs": NL * 2 * 2 * B * S * Hkv * D * 2.0 / (append_us * 1e-6) / 1e9},
                        "attention_all_layers": {"us": layer_us[False], "context": L0, "S": S},
                        "decode_attention_all_layers": {"us": layer_us[True], "context": L0, "S": 1}},
            "attention_per_committed_token": {
                "unit": "us of attention (all layers) per committed token, whole batch",
                "block_diffusion": layer_us[False] / (commits.sum().item() / nsteps),
                "ar_decode": layer_us[True] / B,
                "ratio_ar_over_diffusion": (layer_us[True] / B) / (layer_us[False] / (commits.sum().item() / nsteps)),
                "note": "diffusion: the S=16 attention of every layer per denoise step / the loop's mean commits "
                        "per step; AR: the S=1 attention of every layer per step / B; both at the start context "
                        "length"},
            "gpu_launches": reps * (nsteps * (NL + 1) + NB),   # the timed loops (the other timings are extra)
            "graph": True,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def launches_per_step(cfg) -> int:
    return 2          # one attention kernel + one unmask kernel


def main():
    a = parse()
    cfg = synth.CONFIGS[WORKLOADS[a.config]]
    if a.tau is not None:
        cfg = cfg.replace(tau=a.tau)
    if a.impl == "reference":
        return run_reference(a, cfg)
    if a.config == "loop":
        return run_loop(a, cfg)
    return run_ours(a, cfg)


if __name__ == "__main__":
    sys.exit(main())
