#!/usr/bin/env python3
"""Benchmark of the sparse-MoE NVFP4 layer step on B300.

Default workload: 35B-A3B-shaped decode -- 48 MoE layers, hidden 2048, 256
experts, top-8, expert intermediate 512, batch 1, NVFP4 weights of all experts
resident in HBM, 256 distinct decode steps of synthetic inputs (cycled).  One
bench step = one token through all 48 layers, each layer one fused launch
(router top-k, grouping, NVFP4 SwiGLU expert FFN, weighted combine), replayed
from a CUDA graph per step.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "MoE decode tok/s and % of HBM roofline; prefill NVFP4 TFLOP/s vs peak"
HBM_NOMINAL_GBS = 7700.0  # B300 HBM3e, nominal; the fractions use the measured copy bandwidth, this is context
UNIT = "tok/s"


def load_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    return 1800.0, "fallback"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# --------------------------------------------------------------------------- clocks

class _NvmlLib:
    """The few NVML calls the clock sampler needs, straight from the driver's libnvidia-ml (when the pynvml module
    is not installed).  Read-only: nothing here changes a setting of the GPU."""

    NVML_CLOCK_SM = 1

    def __init__(self, pci_bus_id: str | None):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        rc = (self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) if pci_bus_id
              else self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)))
        if rc != 0:
            raise RuntimeError(f"NVML device handle: error {rc}")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _clock(self, fn) -> int:
        v = self.c.c_uint(0)
        if fn(self.h, self.NVML_CLOCK_SM, self.c.byref(v)) != 0:
            raise RuntimeError("NVML clock query failed")
        return v.value

    def sm_mhz(self) -> int:
        return self._clock(self.lib.nvmlDeviceGetClockInfo)

    def max_sm_mhz(self) -> int:
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def reasons(self) -> int:
        v = self.c.c_ulonglong(0)
        if self.reasons_fn(self.h, self.c.byref(v)) != 0:
            raise RuntimeError("NVML clock-event reasons query failed")
        return v.value


class ClockSampler:
    """Samples SM clock and clock-event reasons while the timed region runs (NVML, else nvidia-smi)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str | None, period_s: float = 0.002):
        self.samples, self.reasons, self.period = [], set(), period_s
        self.max_mhz, self.how, self.err = None, None, None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self.bus = pci_bus_id
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(pci_bus_id) if pci_bus_id
                      else pynvml.nvmlDeviceGetHandleByIndex(0))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.how = "nvml"
        except Exception as e:  # the driver's NVML library directly, else polling nvidia-smi
            self.err = f"{type(e).__name__}: {e}"
            try:
                self.nv = _NvmlLib(pci_bus_id)
                self.h = None
                self.max_mhz = self.nv.max_sm_mhz()
                self.how = "nvml (libnvidia-ml)"
            except Exception as e2:
                self.err += f"; {type(e2).__name__}: {e2}"
                self.how = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        if isinstance(nv, _NvmlLib):
            sm, reasons = nv.sm_mhz, nv.reasons
        else:
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            sm = lambda: nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)  # noqa: E731
            reasons = lambda: fn(self.h)  # noqa: E731
        while True:
            try:
                self.samples.append(sm())
                mask = reasons()
                self.reasons |= {name for bit, name in self.REASONS.items() if mask & bit}
            except Exception as e:
                self.err = f"{type(e).__name__}: {e}"
            if self._stop.is_set():  # one sample after the timed region as well
                break
            time.sleep(self.period)

    def __enter__(self):
        if self.how.startswith("nvml"):
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        else:
            cmd = ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                   "--format=csv,noheader,nounits", "-lms", "50"]
            if self.bus:
                cmd += ["-i", self.bus]
            try:
                self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e:
                self.err = f"{type(e).__name__}: {e}"
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join()
        if self._proc:
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    mask = int(parts[2], 16)
                    self.reasons |= {name for bit, name in self.REASONS.items() if mask & bit}
                except (ValueError, IndexError):
                    pass

    def report(self):
        r = {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
             "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.how}
        if self.err and not self.samples:
            r["error"] = self.err
        return r


# --------------------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int) -> None:
    """One process per GPU: NCCL when CUDA is present, gloo otherwise (the host logic's CPU tests)."""
    if ws > 1:
        import torch
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's time: replicas run independent work, so the job takes as long as its slowest rank."""
    if ws <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


# --------------------------------------------------------------------------- oracle (CPU baseline)

def host_info() -> dict:
    """The host the CPU oracle runs on: CPU model, logical CPUs, and the CPUs this process may use."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        affinity = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        affinity = os.cpu_count()
    return {"cpu_model": model, "nproc": os.cpu_count(), "affinity": affinity}


def single_thread_rate(step, n: int, units_per_step: float, first: int = 20_000) -> float:
    """Units per second of `step` (returns its timed seconds) on one oracle thread over n steps."""
    import oracle as O
    threads = O.lib().ora_max_threads()
    O.set_threads(1)
    try:
        secs = sum(step(first + s) for s in range(n))
    finally:
        O.set_threads(threads)
    return units_per_step * n / secs


class OracleDecode:
    """The CPU oracle on decode steps of one layer of the workload.

    The layer's experts are quantised by the oracle on first use (its inputs,
    untimed); each timed step routes a fresh token, dequantises the selected
    experts, runs their FFN in fp64 and combines -- one layer of one token.
    """

    def __init__(self, cfg: W.MoEConfig, layer: int = 0):
        import oracle as O
        self.O, self.cfg, self.layer = O, cfg, layer
        self.q = {}

    def step(self, s: int) -> float:
        O, cfg = self.O, self.cfg
        logits = W.router_logits(cfg, self.layer, s)
        x_bits = W.activations_bf16(cfg, self.layer, s)
        ids, _ = O.route(logits, cfg.k)
        for e in sorted(set(ids.ravel().tolist())):
            if e not in self.q:
                self.q[e] = [O.quantize_weight(W.weights_fp32(cfg, self.layer, e, p)) for p in range(3)]
        q = self.q

        class _Deq:
            def __init__(self, t):
                self.Wg, self.Wu, self.Wd = (O.dequantize(*a) for a in t)

        t0 = time.perf_counter()
        O.moe_layer(logits, x_bits, cfg.k, lambda e: _Deq(q[e]), O.MODE_A16)
        return time.perf_counter() - t0

    def expert_step(self, s: int) -> float:
        """One routed expert of one token: route, permute, dequantise that expert, its FFN (timed)."""
        O, cfg = self.O, self.cfg
        logits = W.router_logits(cfg, self.layer, s)
        x_bits = W.activations_bf16(cfg, self.layer, s)
        t0 = time.perf_counter()
        ids, w = O.route(logits, cfg.k)
        O.permute(ids, cfg.E)
        t_route = time.perf_counter() - t0
        e = int(ids[0, s % cfg.k])
        if e not in self.q:
            self.q[e] = [O.quantize_weight(W.weights_fp32(cfg, self.layer, e, p)) for p in range(3)]
        x = (x_bits[:1].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        t0 = time.perf_counter()
        Wg, Wu, Wd = (O.dequantize(*a) for a in self.q[e])
        O.expert_ffn(Wg, Wu, Wd, x, O.MODE_A16)
        return t_route + (time.perf_counter() - t0) * cfg.k

    def threads(self) -> int:
        return self.O.lib().ora_max_threads()


REF_BUDGET_S = 60.0  # reference arm: timed oracle seconds after which no further whole step starts


class OracleToken:
    """The CPU oracle on whole decode steps: one token through every layer of the workload (route, permute,
    fp64 dequantisation and FFN of its experts, combine), each layer with its own experts.

    The experts a step needs are drawn and quantised by the oracle before the step (its inputs, untimed), on a
    pool of host threads, and kept for later steps up to a bounded number of them."""

    def __init__(self, cfg: W.MoEConfig, keep: int = 1536):
        import concurrent.futures as cf

        import oracle as O
        self.O, self.cfg, self.keep = O, cfg, keep
        self.q = {}
        self.pool = cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))

    def _quantised(self, layer: int, e: int):
        O, cfg = self.O, self.cfg
        return [O.quantize_weight(W.weights_fp32(cfg, layer, e, p)) for p in range(3)]

    def prepare(self, s: int):
        """Inputs of step s: logits and x of every layer, and the experts it routes to (quantised here)."""
        O, cfg = self.O, self.cfg
        inputs = []
        used, need = [], []
        for layer in range(cfg.layers):
            logits = W.router_logits(cfg, layer, s)
            x_bits = W.activations_bf16(cfg, layer, s)
            ids, _ = O.route(logits, cfg.k)
            inputs.append((logits, x_bits))
            used += [(layer, int(e)) for e in sorted(set(ids.ravel().tolist()))]
        for key in used:  # least recently used first: this step's experts move to the end
            if key in self.q:
                self.q[key] = self.q.pop(key)
            else:
                need.append(key)
        for key, qv in zip(need, self.pool.map(lambda le: self._quantised(*le), need)):
            self.q[key] = qv
        while len(self.q) > max(self.keep, len(used)):  # never evicts this step's experts
            self.q.pop(next(iter(self.q)))
        return inputs

    def step(self, s: int) -> float:
        O, cfg = self.O, self.cfg
        inputs = self.prepare(s)

        class _Deq:
            def __init__(self, t):
                self.Wg, self.Wu, self.Wd = (O.dequantize(*a) for a in t)

        t0 = time.perf_counter()
        for layer, (logits, x_bits) in enumerate(inputs):
            O.moe_layer(logits, x_bits, cfg.k, lambda e, layer=layer: _Deq(self.q[(layer, e)]), O.MODE_A16)
        return time.perf_counter() - t0

    def threads(self) -> int:
        return self.O.lib().ora_max_threads()


def oracle_prefill_baseline(cfg, n_rows: int = 16):
    """The oracle (A4 mode) on a bounded sample of the prefill layer: route and permute all tokens, the expert FFN
    and combine for n_rows tokens; reported as tokens/s and the FLOP rate of that sample."""
    import oracle as O
    logits = W.router_logits(cfg, 0, 0)
    x_bits = W.activations_bf16(cfg, 0, 0)
    q = {}

    class _Deq:
        def __init__(self, t):
            self.Wg, self.Wu, self.Wd = (O.dequantize(*a) for a in t)

    ids, _ = O.route(logits, cfg.k)
    rows = list(range(n_rows))
    for e in sorted(set(ids[rows].ravel().tolist())):
        q[e] = [O.quantize_weight(W.weights_fp32(cfg, 0, e, p)) for p in range(3)]
    t0 = time.perf_counter()
    O.moe_layer(logits, x_bits, cfg.k, lambda e: _Deq(q[e]), O.MODE_A4, rows=np.array(rows))
    secs = time.perf_counter() - t0

    def one_thread_step(s):  # the first two of those tokens again, on one oracle thread
        t1 = time.perf_counter()
        O.moe_layer(logits, x_bits, cfg.k, lambda e: _Deq(q[e]), O.MODE_A4, rows=np.array(rows[:2]))
        return time.perf_counter() - t1

    return {"value": n_rows / secs, "unit": "tok/s", "tflops": 6.0 * cfg.H * cfg.I * cfg.k * n_rows / secs / 1e12,
            "cores": O.lib().ora_max_threads(), "kind": "oracle",
            "sample": f"route and permute of all {cfg.T} tokens, then fp64 dequantisation, A4-mode FFN and combine "
                      f"of {n_rows} tokens (weight quantisation untimed)",
            "single_thread": {"value": single_thread_rate(one_thread_step, 1, 2.0), "unit": "tok/s",
                              "sample": "the same for 2 tokens on one thread"}, **host_info()}


class OraclePrefill:
    """The CPU oracle (A4 mode) on the prefill layer, a few tokens per step: the routing of all T tokens and the
    quantisation of the experts a step needs happen untimed; each timed step runs route, permute, the fp64 expert
    FFN and the combine for `rows` tokens."""

    def __init__(self, cfg, rows: int = 2):
        import oracle as O
        self.O, self.cfg, self.rows = O, cfg, rows
        self.logits = W.router_logits(cfg, 0, 0)
        self.x_bits = W.activations_bf16(cfg, 0, 0)
        self.ids, _ = O.route(self.logits, cfg.k)
        self.q = {}

    def _expert(self, e):
        O = self.O

        class _Deq:
            def __init__(self, t):
                self.Wg, self.Wu, self.Wd = (O.dequantize(*a) for a in t)

        return _Deq(self.q[e])

    def step(self, s: int) -> float:
        T = self.cfg.T
        rows = np.array([(s * self.rows + i) % T for i in range(self.rows)])
        for e in sorted(set(self.ids[rows].ravel().tolist())):
            if e not in self.q:
                self.q[e] = [self.O.quantize_weight(W.weights_fp32(self.cfg, 0, e, p)) for p in range(3)]
        t0 = time.perf_counter()
        self.O.moe_layer(self.logits, self.x_bits, self.cfg.k, self._expert, self.O.MODE_A4, rows=rows)
        return time.perf_counter() - t0

    def threads(self) -> int:
        return self.O.lib().ora_max_threads()


# --------------------------------------------------------------------------- GPU arm

def kernel_source_hash(files=("decode_fused.cu", "common.cuh")) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "quantized_expert_ffn_06_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ("prefill.cu", "route_permute.cu", "common.cuh")


def profiled_traffic(workload: str, src_hash: str, kernel: str = "k_moe_decode", key: str = "dram_bytes_per_launch"):
    """DRAM bytes per launch (or per call) of the measured kernel(s) from the committed ncu summary, if the
    source it was taken on is still the current one."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != src_hash:
        return None
    return d.get(key)


def run_gpu(args, ws, rank, local):
    import torch
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import FusedDecodeLayer, LayerWeights, MoEDecodeLayer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = W.CONFIGS[args.config]
    L, S, T, H, E, k = cfg.layers, min(cfg.steps, args.distinct_steps), cfg.T, cfg.H, cfg.E, cfg.k
    if args.layers:
        L = args.layers
    # the fused layer step stages x and the h rows as f16 in shared memory (120 KB per launch) and runs a
    # larger batch as launches over token chunks that fit; a single token that does not fit takes the
    # separate calls (route, permute, row-layout expert FFN, combine)
    fused = T <= 16 and ((H + 32) + k * (cfg.I + 32)) * 2 <= 120 * 1024
    chunk = max([c for c in range(1, T + 1) if (c * (H + 32) + c * k * (cfg.I + 32)) * 2 <= 120 * 1024] or [1])
    n_chunks = -(-T // chunk)  # launches per layer on the fused path
    layout = Q.FT_LAYOUT_DECODE_TILES if fused else Q.FT_LAYOUT_ROWS
    mx = args.weights in ("mxfp4", "mxfp8")
    if mx:
        if not fused:
            raise SystemExit("MX weights run on the fused decode step only")
        layout = Q.FT_LAYOUT_MXFP4_DECODE_TILES if args.weights == "mxfp4" else Q.FT_LAYOUT_MXFP8_DECODE_TILES
    # bytes of one expert's three matrices: NVFP4 0.5 B per code + 1 B per 16 + three fp32 tensor scales,
    # MXFP4 0.5 B per code + 1 B per 32, MXFP8 1 B per code + 1 B per 32
    expert_bytes = (3 * H * cfg.I * (17 if args.weights == "mxfp4" else 33) // 32 if mx else cfg.expert_bytes + 12)

    # ---- weights (device generator + device quantiser), all experts resident
    weights = []
    for layer in range(L):
        lw = LayerWeights(E, H, cfg.I, dev, layout=layout)
        lw.fill_synthetic(lambda e, p, layer=layer: W.w_stream(cfg.weight_cfg, layer, e, p), sigma=cfg.w_sigma)
        weights.append(lw)
    torch.cuda.synchronize()

    # ---- inputs of S distinct steps, resident in HBM (rank r draws steps offset by r*S)
    step0 = rank * S
    x_host = np.stack([np.stack([W.activations_bf16(cfg, l, step0 + s) for l in range(L)]) for s in range(S)])
    lg_host = np.stack([np.stack([W.router_logits(cfg, l, step0 + s) for l in range(L)]) for s in range(S)])
    x_dev = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).to(dev)     # [S, L, T, H]
    lg_dev = torch.from_numpy(lg_host).to(dev)                                         # [S, L, T, E]
    out_dev = torch.empty((S, L, T, H), dtype=torch.bfloat16, device=dev)

    if fused:
        layer_mods = [FusedDecodeLayer(E, H, cfg.I, k, T, dev) for _ in range(L)]
    else:
        layer_mods = [MoEDecodeLayer(E, H, cfg.I, k, T, dev) for _ in range(L)]
    launches_per_layer = n_chunks if fused else 5  # (route, permute, gate/up, down, combine)
    stream = torch.cuda.Stream(device=dev)

    def step_body(xs, ls, os_):
        for l in range(L):
            if fused:
                layer_mods[l](weights[l], ls[l], xs[l], os_[l], routing=False, stream=stream)
            else:
                layer_mods[l](weights[l], ls[l], xs[l], os_[l], stream=stream)

    # ---- one CUDA graph per distinct step
    with torch.cuda.stream(stream):
        step_body(x_dev[0], lg_dev[0], out_dev[0])   # warm the code paths before capture
    stream.synchronize()
    graphs = []
    for s in range(S):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step_body(x_dev[s], lg_dev[s], out_dev[s])
        graphs.append(g)
    torch.cuda.synchronize()
    assert Q.ft_device_status(stream) == 0

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % S].replay()
    stream.synchronize()

    # ---- timed region: K steps, inputs resident; each step streams ~680 MB of weights (> L2)
    props = torch.cuda.get_device_properties(dev)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(bus) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(args.steps):
                graphs[i % S].replay()
            ev1.record(stream)
        ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, ws, dev)
    value = args.steps * T * ws / (ms / 1e3)
    assert Q.ft_device_status(stream) == 0

    # ---- dominant kernel: the timed region holds only its launches (L per step, back to back in
    # the graph), so its average launch duration is the timed region's CUDA-event span / launches;
    # the gap to the next launch is included
    unique = [len(set(np.argsort(-lg_host[i % S][l], axis=1, kind="stable")[:, :k].ravel().tolist()))
              for i in range(min(args.steps, S)) for l in range(L)]
    # algorithmic bytes of one layer launch: the selected experts' weights (three matrices at 0.5625 B/param
    # plus three fp32 tensor scales for NVFP4, 0.53125 B/param for MXFP4) plus logits, activations and output
    # (with several token chunks per layer, the layer's bytes and time are shared evenly by its launches)
    bytes_per_launch = (float(np.mean(unique)) * expert_bytes + T * (E * 4 + H * 2 * 2)) / (
        n_chunks if fused else 1)
    avg_launch_s = (ms / 1e3) / (args.steps * L * (n_chunks if fused else 1))
    peak, peak_kind = load_peaks()
    achieved = bytes_per_launch / avg_launch_s / 1e9

    # ---- e2e through the public API with pinned host buffers: H2D inputs, layer launches, D2H outputs
    e2e = None
    if not args.no_e2e:
        xb = [torch.empty((L, T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        lb = [torch.empty((L, T, E), dtype=torch.float32, device=dev) for _ in range(2)]
        ob = [torch.empty((L, T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        eg = []
        for j in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_body(xb[j], lb[j], ob[j])
            eg.append(g)
        x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
        l_pin = torch.from_numpy(lg_host).pin_memory()
        o_pin = torch.empty((S, L, T, H), dtype=torch.bfloat16).pin_memory()

        def load_inputs(j, i):
            xb[j].copy_(x_pin[i % S], non_blocking=True)
            lb[j].copy_(l_pin[i % S], non_blocking=True)

        def read_outputs(j, i):
            o_pin[i % S].copy_(ob[j], non_blocking=True)

        barrier()
        ems = run_e2e_pipelined(stream, dev, args.steps, args.warmup, load_inputs, lambda j: eg[j].replay(),
                                read_outputs)
        ems = max_over_ranks(ems, ws, dev)
        e2e = {"value": args.steps * T * ws / (ems / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": L * T * (H * 2 + E * 4), "d2h_bytes_per_step": L * T * H * 2}

    src_hash = kernel_source_hash()
    wfmt = {"mxfp4": "MXFP4 (E2M1 + UE8M0/32)", "mxfp8": "MXFP8 (E4M3 + UE8M0/32)"}.get(
        args.weights, "NVFP4 (E2M1 + E4M3/16 + fp32 tensor scale)")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{args.weights} weights x bf16 activations, fp32 accumulate",
        "data": "synthetic (seeded Philox4x32-10)",
        "config": {"workload": f"{cfg.name}: {L} MoE layers, hidden {H}, {E} experts, top-{k}, intermediate {cfg.I}, "
                               f"batch {T}, {wfmt}, all experts resident",
                   "global_batch": T * ws, "distinct_steps": S,
                   "l2": "inputs larger than L2: each step streams ~%.0f MB of expert weights" %
                         (L * float(np.mean(unique)) * expert_bytes / 1e6),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "nominal_peak": HBM_NOMINAL_GBS,
                     "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
                     "kernel": (("k_moe_decode (ft_moe_layer_decode), one launch per layer" if n_chunks == 1 else
                                 f"k_moe_decode (ft_moe_layer_decode), {n_chunks} launches per layer (token chunks "
                                 f"of {chunk}); the layer's unique-expert bytes and time shared by its launches")
                                if fused else
                                "route + permute + k_decode_gateup + k_decode_down + combine per layer, timed together"),
                     "bytes_per_launch": bytes_per_launch, "avg_launch_us": avg_launch_s * 1e6,
                     "traffic": profiled_traffic(cfg.name + ("_" + args.weights if mx else ""), src_hash) if fused else None,
                     "source_hash": src_hash},
        "e2e": e2e,
        "gpu_launches": L * args.steps * launches_per_layer,
        "clocks": clk.report(),
    }


def run_e2e_pipelined(stream, dev, steps: int, warmup: int, load_inputs, replay, read_outputs) -> float:
    """Milliseconds of `steps` end-to-end steps through two alternating buffer sets: the host -> device copy of
    step i+1's inputs runs on a side stream while step i computes, and step i's result goes device -> host on
    another, so every step's copies stay inside the timed region without serialising with its compute.
    load_inputs(j, i) / read_outputs(j, i) enqueue step i's copies for buffer set j on the current stream;
    replay(j) launches step i's work on it.  Events order every reuse of a buffer set."""
    import torch
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready, in_free = [torch.cuda.Event() for _ in range(2)], [torch.cuda.Event() for _ in range(2)]
    out_ready, out_free = [torch.cuda.Event() for _ in range(2)], [torch.cuda.Event() for _ in range(2)]

    def issue_inputs(i):
        j = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(in_free[j])    # the step that last read buffer set j has finished
            load_inputs(j, i)
            in_ready[j].record(h2d)

    def run(n):
        h2d.wait_stream(stream)
        issue_inputs(0)
        for i in range(n):
            j = i % 2
            if i + 1 < n:
                issue_inputs(i + 1)
            with torch.cuda.stream(stream):
                stream.wait_event(in_ready[j])
                stream.wait_event(out_free[j])   # the previous result in buffer set j has reached the host
                replay(j)
                in_free[j].record(stream)
                out_ready[j].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(out_ready[j])
                read_outputs(j, i)
                out_free[j].record(d2h)
        stream.wait_stream(d2h)

    run(warmup)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def prefill_launches(T: int, k: int) -> int:
    """Kernels one prefill layer step launches: the router, the permutation (one block up to 1024 routed pairs,
    else histogram + scan + placement) and the FFN call (plan, x quantisation, gather, two GEMMs, output)."""
    return 1 + (1 if T * k <= 1024 else 3) + 6


def bench_config(args):
    """The named workload; for a prefill workload ``--tokens`` sets the prompt length of a T-sweep point."""
    cfg = W.CONFIGS[args.config]
    if args.tokens:
        if cfg.routing != "zipf":
            raise SystemExit("--tokens applies to the prefill workload only")
        cfg = W.scaled(cfg, T=args.tokens, name=f"{cfg.name}_t{args.tokens}")
    return cfg


def run_gpu_prefill(args, ws, rank, local):
    """Prefill layer step: T tokens through route -> permute -> tensor-core NVFP4 expert FFN + combine."""
    import torch
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import LayerWeights, PrefillLayer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = bench_config(args)
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    NW = 4  # weight sets rotated between steps: 4 x the layer's weights, far beyond L2
    S = min(args.distinct_steps, 4)
    if args.weights == "mxfp8":
        raise SystemExit("the tensor-core prefill takes NVFP4 or MXFP4 weights")
    mx4 = args.weights == "mxfp4"  # MXFP4 re-encoded exactly into the FP4 tensor-core tiles
    weights = []
    for l in range(NW):
        lw = LayerWeights(E, H, I, dev, layout=Q.FT_LAYOUT_UMMA_TILES, source=args.weights)
        lw.fill_synthetic(lambda e, p, l=l: W.w_stream(cfg.weight_cfg, l, e, p), sigma=cfg.w_sigma)
        weights.append(lw)
    step0 = rank * S
    lg_host = np.stack([W.router_logits(cfg, s % NW, step0 + s) for s in range(S)])
    x_host = np.stack([W.activations_bf16(cfg, s % NW, step0 + s) for s in range(S)])
    lg_dev = torch.from_numpy(lg_host).to(dev)
    x_dev = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    mod = PrefillLayer(E, H, I, k, T, dev)
    stream = torch.cuda.Stream(device=dev)
    n_cfg = NW * S  # (weight set, input) pairs cycled by the steps
    with torch.cuda.stream(stream):
        mod(weights[0], lg_dev[0], x_dev[0], out, stream=stream)
    stream.synchronize()
    graphs = []
    for i in range(n_cfg):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            mod(weights[i % NW], lg_dev[i % S], x_dev[i % S], out, stream=stream)
        graphs.append(g)
    torch.cuda.synchronize()
    assert Q.ft_device_status(stream) == 0
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % n_cfg].replay()
    stream.synchronize()
    props = torch.cuda.get_device_properties(dev)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(bus) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(args.steps):
                graphs[i % n_cfg].replay()
            ev1.record(stream)
        ev1.synchronize()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, ws, dev)
    assert Q.ft_device_status(stream) == 0
    step_s = ms / 1e3 / args.steps
    # the expert FFN call alone (its kernels: plan, x quantisation, two grouped GEMMs, output), live, same stream
    fe0, fe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_ffn = max(8, min(args.steps, 64))
    with torch.cuda.stream(stream):
        for i in range(n_cfg):
            mod(weights[i % NW], lg_dev[i % S], x_dev[i % S], out, stream=stream)
        fe0.record(stream)
        for i in range(n_ffn):
            Q.ft_moe_expert_ffn_nvfp4_prefill(weights[i % NW], x_dev[0], k, mod.offsets, mod.perm, mod.w, out, mod.ws,
                                              stream=stream)
        fe1.record(stream)
    stream.synchronize()
    ffn_s = fe0.elapsed_time(fe1) / 1e3 / n_ffn
    # algorithmic work: real (unpadded) FLOPs 2*3*H*I per routed row; bytes = weights of the experts that
    # received rows + x + logits + output
    P = T * k
    flops = 6.0 * H * I * P
    touched = np.mean([len(set(np.argsort(-lg_host[s], axis=1, kind="stable")[:, :k].ravel().tolist()))
                       for s in range(S)])
    bytes_ffn = touched * (cfg.expert_bytes + 12) + T * H * 2 * 2
    hbm_peak, hbm_kind = load_peaks()
    bf16_peak, bf16_kind = load_bf16_peak()
    fp4_peak = bf16_peak * 6.0  # nominal dense FP4 : BF16 ratio of 13.5 : 2.25
    ai = flops / bytes_ffn  # FLOP per algorithmic byte
    attainable = min(fp4_peak, hbm_peak * ai / 1e3)  # TFLOP/s
    e2e = None
    if not args.no_e2e:
        x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
        l_pin = torch.from_numpy(lg_host).pin_memory()
        o_pin = torch.empty((2, T, H), dtype=torch.bfloat16).pin_memory()
        xb = [torch.empty_like(x_dev[0]) for _ in range(2)]
        lb = [torch.empty_like(lg_dev[0]) for _ in range(2)]
        ob = [torch.empty_like(out) for _ in range(2)]
        eg = {}
        for i in range(NW):  # a graph per (weight set, buffer set); step i uses weight set i % NW
            for j in range(2):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    mod(weights[i], lb[j], xb[j], ob[j], stream=stream)
                eg[i, j] = g
        step_of = [0, 0]  # the step each buffer set currently carries

        def load_inputs(j, i):
            step_of[j] = i
            xb[j].copy_(x_pin[i % S], non_blocking=True)
            lb[j].copy_(l_pin[i % S], non_blocking=True)

        def read_outputs(j, i):
            o_pin[j].copy_(ob[j], non_blocking=True)

        ems = run_e2e_pipelined(stream, dev, args.steps, args.warmup, load_inputs,
                                lambda j: eg[step_of[j] % NW, j].replay(), read_outputs)
        ems = max_over_ranks(ems, ws, dev) / 1e3 / args.steps
        e2e = {"value": flops / ems / 1e12, "unit": "TFLOP/s", "tok_per_s": T / ems,
               "h2d_bytes_per_step": T * (H * 2 + E * 4), "d2h_bytes_per_step": T * H * 2}
    return {
        "metric": METRIC, "value": flops * ws / step_s / 1e12, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("mxfp4 weights (UE8M0 per 32, re-encoded exactly as power-of-two UE4M3 per 16) x nvfp4 activations, "
                  "fp32 accumulate" if mx4 else "nvfp4 x nvfp4 (E2M1, UE4M3 per 16), fp32 accumulate"),
        "data": "synthetic (seeded Philox4x32-10, Zipf(1.1) expert popularity)",
        "tok_per_s": T * ws / step_s,
        "config": {"workload": f"{cfg.name}: one MoE layer, hidden {H}, {E} experts, top-{k}, intermediate {I}, "
                               f"{T} prompt tokens, " + ("MXFP4 weights, NVFP4 activations" if mx4 else
                                                         "NVFP4 weights and activations"),
                   "global_batch": T * ws,
                   "l2": f"inputs larger than L2: {NW} weight sets of {touched * cfg.expert_bytes / 1e6:.0f} MB "
                         f"rotated between steps",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": bytes_ffn / ffn_s / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": bytes_ffn / ffn_s / 1e9 / hbm_peak, "peak_kind": hbm_kind,
                     "kernel": "ft_moe_expert_ffn_nvfp4_prefill (plan, x quantisation, gate/up and down grouped "
                               "GEMMs, output), timed as one call",
                     "bytes_per_launch": bytes_ffn, "avg_launch_us": ffn_s * 1e6,
                     "traffic": profiled_traffic(cfg.name + ("_mxfp4" if mx4 else ""),
                                                 kernel_source_hash(PREFILL_SOURCES), "k_pf_ffn", "dram_bytes_per_call"),
                     "traffic_what": "DRAM bytes read + written by the FFN call's kernels (plan, x quantisation, "
                                     "gather, both GEMMs, output), from the committed ncu launch list"},
        "attainable": {"tflops": attainable, "frac": flops / ffn_s / 1e12 / attainable,
                       "bound": "hbm" if hbm_peak * ai / 1e3 < fp4_peak else "tensor", "flop_per_byte": ai,
                       "what": "the FFN call against min(FP4 peak, HBM peak x its arithmetic intensity)"},
        "tensor": {"achieved": flops / ffn_s / 1e12, "peak": fp4_peak, "unit": "TFLOP/s",
                   "frac": flops / ffn_s / 1e12 / fp4_peak,
                   "peak_kind": f"{bf16_kind} bf16 x 6 (nominal FP4:BF16 dense ratio)", "flops_per_launch": flops},
        "e2e": e2e,
        "gpu_launches": args.steps * prefill_launches(T, k),
        "clocks": clk.report(),
    }


def run_gpu_prefill_stream(args, ws, rank, local):
    """Prefill through L layers whose experts stream from pinned host memory, double-buffered: layer l+1's experts
    copy host -> device on a side stream while layer l computes (per-layer inputs are independent draws)."""
    import torch
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import LayerWeights, StreamedPrefill

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = bench_config(args)
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    if args.weights != "nvfp4":
        raise SystemExit("--stream-layers streams NVFP4 layers")
    L = args.stream_layers
    sp = StreamedPrefill(L, E, H, I, k, T, dev)
    scratch = LayerWeights(E, H, I, dev, layout=Q.FT_LAYOUT_UMMA_TILES)
    for l in range(L):
        scratch.fill_synthetic(lambda e, p, l=l: W.w_stream(cfg.weight_cfg, l, e, p), sigma=cfg.w_sigma)
        sp.load_layer(l, scratch)
    del scratch
    lg_host = [W.router_logits(cfg, l, rank) for l in range(L)]
    lg_dev = [torch.from_numpy(a).to(dev) for a in lg_host]
    x_dev = [torch.from_numpy(W.activations_bf16(cfg, l, rank).view(np.int16)).view(torch.bfloat16).to(dev)
             for l in range(L)]
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    stream = torch.cuda.Stream(device=dev)
    # the two sides of the pipeline alone: one layer's copy, and one layer's compute on resident weights
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        sp.bufs[0].copy_(sp.host[:sp.layer_bytes], non_blocking=True)
        c0.record(stream)
        for l in range(4):
            sp.bufs[0].copy_(sp.host[(l % L) * sp.layer_bytes:(l % L + 1) * sp.layer_bytes], non_blocking=True)
        c1.record(stream)
    torch.cuda.synchronize()
    copy_s = c0.elapsed_time(c1) / 1e3 / 4
    sp.bufs[0].copy_(sp.host[:sp.layer_bytes])
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            sp.layer(sp.buffer_weights(0), lg_dev[0], x_dev[0], outs[0], stream=stream)
        c0.record(stream)
        for _ in range(8):
            sp.layer(sp.buffer_weights(0), lg_dev[0], x_dev[0], outs[0], stream=stream)
        c1.record(stream)
    torch.cuda.synchronize()
    comp_s = c0.elapsed_time(c1) / 1e3 / 8
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            sp(lg_dev, x_dev, outs, stream=stream)
    torch.cuda.synchronize()
    assert Q.ft_device_status(stream) == 0
    props = torch.cuda.get_device_properties(dev)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(bus) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                sp(lg_dev, x_dev, outs, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, ws, dev)
    assert Q.ft_device_status(stream) == 0
    step_s = ms / 1e3 / args.steps
    flops = 6.0 * H * I * T * k * L
    # pipeline bound: the slower side for every layer, plus the faster side once (the first copy, the last layer)
    bound_s = L * max(copy_s, comp_s) + min(copy_s, comp_s)
    return {
        "metric": METRIC, "value": flops * ws / step_s / 1e12, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 x nvfp4 (E2M1, UE4M3 per 16), fp32 accumulate",
        "data": "synthetic (seeded Philox4x32-10, Zipf(1.1) expert popularity)",
        "tok_per_s": T * ws / step_s,
        "config": {"workload": f"{cfg.name}: {L} MoE layers streamed from pinned host memory (double-buffered), "
                               f"hidden {H}, {E} experts, top-{k}, intermediate {I}, {T} prompt tokens per layer",
                   "global_batch": T * ws, "l2": f"inputs larger than L2: {L} layers of {sp.layer_bytes / 1e6:.0f} MB "
                                                f"copied from host every step",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "pcie+tensor", "achieved": 1.0 / step_s, "peak": 1.0 / bound_s, "unit": "steps/s",
                     "frac": bound_s / step_s,
                     "peak_kind": f"measured: one layer's H2D copy {copy_s * 1e3:.2f} ms "
                                  f"({sp.layer_bytes / copy_s / 1e9:.1f} GB/s pinned), one layer's compute on resident "
                                  f"weights {comp_s * 1e3:.3f} ms",
                     "kernel": "L layers: H2D weight copy on a side stream overlapped with route, permute and the "
                               "tensor-core FFN of the previous layer",
                     "copy_ms_per_layer": copy_s * 1e3, "compute_ms_per_layer": comp_s * 1e3,
                     "serial_ms": L * (copy_s + comp_s) * 1e3, "traffic": None},
        "e2e": None,
        "gpu_launches": args.steps * L * prefill_launches(T, k),
        "clocks": clk.report(),
    }


def run_gpu_cache(args, ws, rank, local):
    """Expert-cache decode stream: batch-1 tokens through L layers whose experts live in pinned host memory, with a
    VRAM LRU cache of S slots per layer (misses filled by cudaMemcpyAsync on a side stream)."""
    import torch
    import quantized_expert_ffn_06_b300 as Q
    from quantized_expert_ffn_06_b300.layer import CachedDecodeLayer, ExpertSlotPool, LayerWeights

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = W.CONFIGS[args.config]
    L, T, H, E, k, I = cfg.layers, cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    if args.layers:
        L = args.layers
    n_steps = args.warmup + args.steps
    pool = ExpertSlotPool(L, E, H, I, cfg.slots, dev)
    scratch = LayerWeights(E, H, I, dev, layout=Q.FT_LAYOUT_DECODE_TILES)
    for l in range(L):
        scratch.fill_synthetic(lambda e, p, l=l: W.w_stream(cfg.weight_cfg, l, e, p), sigma=cfg.w_sigma)
        pool.load_layer(l, scratch)
    del scratch
    torch.cuda.synchronize()
    # routing of every (layer, step); activations cycle over 16 distinct draws (they do not affect the routing)
    rank_off = rank * n_steps
    lg_dev = torch.stack([torch.from_numpy(W.cache_stream_logits(cfg, l, rank_off + n_steps)[rank_off:])
                          for l in range(L)]).to(dev)                                   # [L, steps, E]
    NX = 16
    x_dev = torch.from_numpy(np.stack([np.stack([W.activations_bf16(cfg, l, s) for l in range(L)])
                                       for s in range(NX)]).view(np.int16)).view(torch.bfloat16).to(dev)  # [NX, L, T, H]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    stream = torch.cuda.Stream(device=dev)
    P = args.prefetch
    layers = [CachedDecodeLayer(pool, l, k, T, copy_stream=copy_stream,
                                prefetch=P if args.prefetch_source == "router" else 0) for l in range(L)]
    # pinned host -> device copy bandwidth on this machine (the bound of the misses)
    probe_h = torch.empty(512 << 20, dtype=torch.uint8, pin_memory=True)
    probe_d = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    probe_d.copy_(probe_h, non_blocking=True)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    for _ in range(4):
        probe_d.copy_(probe_h, non_blocking=True)
    p1.record()
    torch.cuda.synchronize()
    h2d_gbs = 4 * (512 << 20) / (p0.elapsed_time(p1) / 1e3) / 1e9
    del probe_h, probe_d

    # predictions: the router's next P ranks (the mechanism), or the next token's own experts (an exact
    # predictor: the bound on what prefetching can save on this stream)
    exact = args.prefetch_source == "next"
    nxt = [W.cache_stream_sets(cfg, l, rank_off + n_steps + 1)[rank_off:] for l in range(L)] if exact else None

    def token(s):
        for l in range(L):
            layers[l](lg_dev[l, s][None, :], x_dev[s % NX, l], out, rank_off + s, stream=stream,
                      predicted=nxt[l][s + 1] if exact else None)

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            token(s)
    torch.cuda.synchronize()
    h0, m0, b0 = pool.cache.stats()
    pf0, pu0 = pool.cache.prefetch_stats()
    for lay in layers:
        lay.host_wait_s = lay.host_cache_s = lay.host_call_s = 0.0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(bus) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for s in range(args.warmup, n_steps):
                token(s)
            e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, ws, dev)
    assert Q.ft_device_status(stream) == 0
    h1, m1, b1 = pool.cache.stats()
    hits, misses, filled = h1 - h0, m1 - m0, b1 - b0
    pf1, pu1 = pool.cache.prefetch_stats()
    prefetched, used = pf1 - pf0, pu1 - pu0
    step_s = ms / 1e3 / args.steps
    hbm_peak, hbm_kind = load_peaks()
    # elastic resize at a safe point, after the timed stream: every layer shrinks to half its slots in a new pool
    # (the most recently used half moves device to device), then grows back (all of them move again)
    resize = {}
    S0 = pool.S
    for name, n in (("shrink", S0 // 2), ("grow", S0)):
        moved = sum(q >= 0 for row in pool.cache.resize_plan(n) for q in row)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        r0.record(stream)
        pool.resize(n, stream=stream)
        r1.record(stream)
        torch.cuda.synchronize()
        t_s = r0.elapsed_time(r1) / 1e3
        resize[name] = {"slots": f"{S0 if name == 'shrink' else S0 // 2} -> {n} per layer", "experts_moved": moved,
                        "bytes_moved": moved * pool.expert_bytes, "ms": t_s * 1e3,
                        "gbs_read_plus_write": 2 * moved * pool.expert_bytes / t_s / 1e9,
                        "frac_of_hbm_copy": 2 * moved * pool.expert_bytes / t_s / 1e9 / hbm_peak}
    assert Q.ft_device_status(stream) == 0
    # per-token bound: every layer must bring its misses over PCIe and stream its k experts from HBM
    miss_bytes_tok = filled / args.steps
    hbm_bytes_tok = L * k * pool.expert_bytes
    bound_s = miss_bytes_tok / (h2d_gbs * 1e9) + hbm_bytes_tok / (hbm_peak * 1e9)
    return {
        "metric": METRIC, "value": T * ws / step_s, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 weights x bf16 activations, fp32 accumulate",
        "data": "synthetic (seeded Philox4x32-10; Zipf(1.1) popularity, 60 % of experts shared between tokens)",
        "config": {"workload": f"{cfg.name}: {L} MoE layers, hidden {H}, {E} experts, top-{k}, intermediate {I}, "
                               f"batch {T}, VRAM LRU cache of {cfg.slots} slots per layer over a "
                               f"{L * E * pool.slot_stride / 1e9:.1f} GB pinned host pool"
                               + (f", router-driven prefetch of the next {P} ranks" if P and not exact else "")
                               + (", prefetch of the next token's experts (exact predictor)" if exact else ""),
                   "global_batch": T * ws, "l2": "inputs larger than L2: misses come from host memory",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "cache": {"hit_rate": hits / max(1, hits + misses), "hits": hits, "misses": misses,
                  "h2d_bytes_per_token": miss_bytes_tok, "h2d_gbs_achieved": filled / (ms / 1e3) / 1e9,
                  "h2d_gbs_measured_peak": h2d_gbs,
                  "host_ms_per_token": {
                      "routing_wait": sum(lay.host_wait_s for lay in layers) * 1e3 / args.steps,
                      "cache_logic": sum(lay.host_cache_s for lay in layers) * 1e3 / args.steps,
                      "enqueue": sum(lay.host_call_s for lay in layers) * 1e3 / args.steps,
                      "what": "host wall time per token, all layers: waiting for each layer's routing result (the "
                              "device work queued before it: the previous layers' kernels and copies), the cache's "
                              "host logic (lookup, fill and prefetch enqueues, publish), and the route/kernel "
                              "launches"},
                  "prefetch": {"next_ranks": P, "source": args.prefetch_source, "prefetched": prefetched, "used": used,
                               "accuracy": used / prefetched if prefetched else None,
                               "demand_misses_per_token": misses / args.steps,
                               "what": "predicted experts (source router: the router's next P ranks of each token; "
                                       "source next: the next token's own experts, an exact predictor) installed "
                                       "for the next token and copied behind its misses on the copy stream; "
                                       "accuracy = installed experts a later lookup found / installed"},
                  "resize": dict(resize, what="ft_expert_cache_resize after the timed stream (device-to-device "
                                              "moves + the publish of every layer's table), CUDA events on the "
                                              "stream; not part of the tok/s")},
        "roofline": {"bound": "pcie+hbm", "achieved": 1.0 / step_s, "peak": 1.0 / bound_s, "unit": "tok/s",
                     "frac": bound_s / step_s, "peak_kind": f"measured pinned H2D {h2d_gbs:.1f} GB/s and {hbm_kind} HBM",
                     "kernel": "whole token (route, host lookup, fills, slot-table publish, fused layer kernel) x layers",
                     "traffic": None},
        "e2e": None,
        "gpu_launches": L * args.steps * 2,
        "clocks": clk.report(),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode_35b")
    ap.add_argument("--distinct-steps", type=int, default=256)
    ap.add_argument("--layers", type=int, default=0, help="(debug) fewer layers; the result is then not the workload")
    ap.add_argument("--prefetch-source", default="router", choices=["router", "next"],
                    help="cache stream: predictions from the router's ranks, or the next token's experts (exact)")
    ap.add_argument("--weights", default="nvfp4", choices=["nvfp4", "mxfp4", "mxfp8"],
                    help="expert weight format: decode configs (fused layer step) and the prefill workload (nvfp4, mxfp4)")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="cache stream: install the router's next P ranked experts of each token for the next one")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode_35b: skip the prefill measurement reported beside the decode line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-steps", type=int, default=48)
    ap.add_argument("--stream-layers", type=int, default=0,
                    help="prefill only: that many layers streamed from pinned host memory, double-buffered")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prefill only: prompt tokens per step instead of the workload's 4096 (a labelled T-sweep point)")
    args = ap.parse_args()

    ws, rank, local = dist_env()
    cfg = bench_config(args)

    if args.impl == "reference":
        if rank != 0:
            return
        if cfg.routing == "zipf":
            # the prefill workload: the oracle's FLOP rate on a few tokens per step, in the GPU arm's unit
            ref = OraclePrefill(cfg)
            for s in range(args.warmup):
                ref.step(10_000 + s)
            secs = sum(ref.step(s) for s in range(args.steps))
            flops = 6.0 * cfg.H * cfg.I * cfg.k * ref.rows * args.steps
            val = flops / secs / 1e12
            layer_ms = secs / (ref.rows * args.steps) * cfg.T * 1e3
            line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": 1,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_step": layer_ms, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                    "data": "synthetic (seeded Philox4x32-10, Zipf(1.1) expert popularity)",
                    "config": {"workload": cfg.name},
                    "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": ref.threads(), "kind": "oracle",
                                     "sample": f"each step: route and permute of all {cfg.T} tokens, then the fp64 "
                                               f"A4-mode expert FFN and combine of {ref.rows} tokens (expert "
                                               f"quantisation untimed); ms_per_step scales that to {cfg.T} tokens"},
                    "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(line))
            return
        # the oracle as it stands on the host cores, on whole steps: one token through all the layers; the timed
        # steps stop early (whole steps, at least one) once they have taken REF_BUDGET_S, so that a run asked for
        # many steps still ends within minutes; "steps" is the number timed, "steps_requested" the number asked
        ref = OracleToken(cfg)
        for s in range(args.warmup):
            ref.step(10_000 + s)
        secs, done = 0.0, 0
        while done < args.steps and (done == 0 or secs < REF_BUDGET_S):
            secs += ref.step(done)
            done += 1
        per_token = secs / done
        val = cfg.T / per_token
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1, "steps": done,
                "steps_requested": args.steps,
                "warmup": args.warmup, "ms_per_step": per_token * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Philox4x32-10)",
                "config": {"workload": cfg.name},
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": ref.threads(), "kind": "oracle",
                                 "sample": f"each step: one token through all {cfg.layers} layers (route, permute, "
                                           f"fp64 dequantisation and FFN of its {cfg.k} experts per layer, combine); "
                                           f"drawing and quantising the experts untimed"},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    init_dist(ws)
    if cfg.routing == "stream":
        res = run_gpu_cache(args, ws, rank, local)
        if rank == 0:
            print(json.dumps(res))
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    if cfg.routing == "zipf" and args.stream_layers:
        res = run_gpu_prefill_stream(args, ws, rank, local)
        if rank == 0:
            print(json.dumps(res))
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    if cfg.routing == "zipf":
        res = run_gpu_prefill(args, ws, rank, local)
        if rank == 0:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = oracle_prefill_baseline(cfg)
            print(json.dumps(res))
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    res = run_gpu(args, ws, rank, local)
    if args.config == "decode_35b" and not args.no_prefill and args.weights != "mxfp8":  # no MXFP8 prefill path
        # the same layer shape's 4096-token prefill (grouped FP4 tensor-core GEMMs), measured in the same run
        # after the decode and reported beside it: its own workload, unit and roofline
        import argparse as _ap
        pa = _ap.Namespace(**vars(args))
        pa.config, pa.steps, pa.warmup, pa.tokens = "prefill_35b", 20, 5, 0
        pres = run_gpu_prefill(pa, ws, rank, local)
        res["prefill"] = {key: pres[key] for key in ("metric", "value", "unit", "ms_per_step", "steps", "warmup",
                                                     "dtype", "config", "roofline", "e2e", "gpu_launches", "clocks")
                          if key in pres}
    if rank == 0:
        if not args.no_cpu_baseline:
            ref = OracleDecode(cfg)
            secs = sum(ref.step(s) for s in range(args.cpu_steps))
            per_token = secs / args.cpu_steps * cfg.layers
            res["cpu_baseline"] = {"value": cfg.T / per_token, "unit": UNIT, "cores": ref.threads(), "kind": "oracle",
                                   "sample": f"{args.cpu_steps} single-token steps of layer 0 (route, permute, fp64 "
                                             f"dequantisation, FFN, combine), scaled to {cfg.layers} layers; "
                                             f"weight generation and quantisation untimed",
                                   "single_thread": {"value": single_thread_rate(ref.step, 4, cfg.T / cfg.layers),
                                                     "unit": UNIT, "sample": "4 such steps on one thread"},
                                   **host_info()}
        print(json.dumps(res))
    if ws > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
