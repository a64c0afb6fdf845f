"""Seeded synthetic workloads for the sparse-MoE layer step.

This package is shared by the CUDA path's tests and benchmark and by the CPU
oracle, and by design holds none of the method's arithmetic: it draws weights,
activations and router logits, nothing else.  Every number comes from the
counter-based Philox4x32-10 generator (Salmon et al., SC'11) in ``ftgen.c``,
addressed by (seed, stream, index), so any slice of any tensor can be
regenerated on its own.

Stream identifiers (64 bit):

* weights   ``1<<56 | cfg<<48 | layer<<32 | expert<<8 | proj``  (proj 0 gate, 1 up, 2 down),
  element index ``n*K + k`` of the fp32 matrix ``[N, K]``;
* activations ``2<<56 | cfg<<48 | layer<<32 | step``, index ``t*H + h``;
* router logits ``3<<56 | cfg<<48 | layer<<32 | step``, index ``t*E + e``;
* Zipf rank map ``4<<56 | cfg<<48 | layer<<32``; Gumbel noise ``5<<56 | ...``;
* cache-stream draws ``6<<56 | cfg<<48 | layer<<32 | step<<4 | what``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ftgen.c")
_LIB = os.path.join(_HERE, "libftgen.so")
_lock = threading.Lock()
_lib = None

SEED = 0
PROJ_GATE, PROJ_UP, PROJ_DOWN = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ftgen.c into workloads/libftgen.so (plain gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            L.ftgen_philox4x32_10.argtypes = [vp, vp, vp]
            L.ftgen_uniform_f64.argtypes = [u64, u64, u64, i64, vp]
            L.ftgen_normal_f32.argtypes = [u64, u64, u64, i64, dbl, vp]
            L.ftgen_normal_f64.argtypes = [u64, u64, u64, i64, dbl, vp]
            L.ftgen_normal_bf16.argtypes = [u64, u64, u64, i64, dbl, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ---------------------------------------------------------------------------
# raw streams
# ---------------------------------------------------------------------------

def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().ftgen_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(stream: int, n: int, first: int = 0, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        lib().ftgen_uniform_f64(seed, stream, first, n, _ptr(out))
    return out


def normal_f32(stream: int, n: int, sigma: float = 1.0, first: int = 0, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    if n:
        lib().ftgen_normal_f32(seed, stream, first, n, sigma, _ptr(out))
    return out


def normal_f64(stream: int, n: int, sigma: float = 1.0, first: int = 0, seed: int = SEED) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        lib().ftgen_normal_f64(seed, stream, first, n, sigma, _ptr(out))
    return out


def normal_bf16(stream: int, n: int, sigma: float = 1.0, first: int = 0, seed: int = SEED) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0,1), rounded to nearest even from fp32."""
    out = np.empty(n, dtype=np.uint16)
    if n:
        lib().ftgen_normal_bf16(seed, stream, first, n, sigma, _ptr(out))
    return out


def w_stream(cfg: int, layer: int, expert: int, proj: int) -> int:
    return (1 << 56) | (cfg << 48) | (layer << 32) | (expert << 8) | proj


def x_stream(cfg: int, layer: int, step: int) -> int:
    return (2 << 56) | (cfg << 48) | (layer << 32) | step


def logit_stream(cfg: int, layer: int, step: int) -> int:
    return (3 << 56) | (cfg << 48) | (layer << 32) | step


def zipf_map_stream(cfg: int, layer: int) -> int:
    return (4 << 56) | (cfg << 48) | (layer << 32)


def gumbel_stream(cfg: int, layer: int, step: int) -> int:
    return (5 << 56) | (cfg << 48) | (layer << 32) | step


def cache_stream(cfg: int, layer: int, step: int, what: int) -> int:
    return (6 << 56) | (cfg << 48) | (layer << 32) | (step << 4) | what


# ---------------------------------------------------------------------------
# workload shapes
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class MoEConfig:
    """One synthetic workload: layer shape, tokens per step, layers, steps and routing recipe."""

    name: str
    H: int          # hidden size
    I: int          # expert intermediate size
    E: int          # number of experts
    k: int          # experts per token
    T: int          # tokens per step (batch for decode, prompt length for prefill)
    layers: int
    steps: int
    cfg_id: int     # stream namespace for activations and logits
    weight_cfg: int  # stream namespace for weights (shared by decode and prefill of one model shape)
    routing: str = "normal"  # "normal" | "zipf" | "stream"
    w_sigma: float = 0.02
    slots: int = 0           # expert-cache slots per layer (cache stream only)
    share: float = 0.0       # probability of keeping each previous expert (cache stream only)
    zipf_s: float = 1.1

    @property
    def expert_bytes(self) -> int:
        """NVFP4 bytes of one expert: three matrices of H*I elements at 0.5 B + 1 B per 16."""
        return 3 * (self.H * self.I // 2 + self.H * self.I // 16)

    def weight_shape(self, proj: int):
        return (self.I, self.H) if proj in (PROJ_GATE, PROJ_UP) else (self.H, self.I)


CONFIGS = {
    # tiny single layer, every output checked
    "tiny": MoEConfig("tiny", H=256, I=128, E=8, k=2, T=4, layers=1, steps=1, cfg_id=1, weight_cfg=1),
    # 35B-A3B-shaped decode, batch 1, 48 layers, 256 steps, all experts resident
    "decode_35b": MoEConfig("decode_35b", H=2048, I=512, E=256, k=8, T=1, layers=48, steps=256,
                            cfg_id=2, weight_cfg=2),
    # same layer shape, 4096-token prefill with Zipf(1.1) expert popularity
    "prefill_35b": MoEConfig("prefill_35b", H=2048, I=512, E=256, k=8, T=4096, layers=1, steps=1,
                             cfg_id=3, weight_cfg=2, routing="zipf"),
    # 753B-class-shaped decode, 16 layers, 128 steps, batch 1 and batch 16
    "decode_753b_b1": MoEConfig("decode_753b_b1", H=6144, I=2048, E=256, k=8, T=1, layers=16, steps=128,
                                cfg_id=4, weight_cfg=4),
    "decode_753b_b16": MoEConfig("decode_753b_b16", H=6144, I=2048, E=256, k=8, T=16, layers=16, steps=128,
                                 cfg_id=4, weight_cfg=4),
    # expert-cache decode stream: 32 layers, 512 steps, 25% of experts cached per layer
    "cache_stream": MoEConfig("cache_stream", H=4096, I=1536, E=128, k=8, T=1, layers=32, steps=512,
                              cfg_id=5, weight_cfg=5, routing="stream", slots=32, share=0.6),
}


def scaled(cfg: MoEConfig, **kw) -> MoEConfig:
    return replace(cfg, **kw)


# ---------------------------------------------------------------------------
# tensors
# ---------------------------------------------------------------------------

def weights_fp32(cfg: MoEConfig, layer: int, expert: int, proj: int) -> np.ndarray:
    """fp32 matrix [N, K] ~ N(0, w_sigma): gate/up are [I, H], down is [H, I]."""
    N, K = cfg.weight_shape(proj)
    return normal_f32(w_stream(cfg.weight_cfg, layer, expert, proj), N * K, cfg.w_sigma).reshape(N, K)


def activations_bf16(cfg: MoEConfig, layer: int, step: int, T: int | None = None) -> np.ndarray:
    """bf16 bit patterns [T, H] of N(0,1) activations."""
    T = cfg.T if T is None else T
    return normal_bf16(x_stream(cfg.cfg_id, layer, step), T * cfg.H, 1.0).reshape(T, cfg.H)


def zipf_popularity(cfg: MoEConfig, layer: int) -> np.ndarray:
    """p_e for each expert: p_rank ∝ rank^-s, ranks assigned to experts by a seeded permutation."""
    ranks = np.arange(1, cfg.E + 1, dtype=np.float64)
    p_rank = ranks ** (-cfg.zipf_s)
    p_rank /= p_rank.sum()
    order = np.argsort(uniform(zipf_map_stream(cfg.cfg_id, layer), cfg.E), kind="stable")
    p = np.empty(cfg.E)
    p[order] = p_rank          # expert order[r] has rank r+1
    return p


def gumbel(stream: int, n: int) -> np.ndarray:
    u = uniform(stream, n) + 2.0 ** -54   # strictly inside (0, 1)
    return -np.log(-np.log(u))


def router_logits(cfg: MoEConfig, layer: int, step: int, T: int | None = None) -> np.ndarray:
    """fp32 router logits [T, E].

    normal: N(0,1).  zipf: log p_e + Gumbel(0,1), so that top-k draws experts
    without replacement in proportion to p (Gumbel-top-k).
    """
    T = cfg.T if T is None else T
    if cfg.routing == "zipf":
        p = zipf_popularity(cfg, layer)
        g = gumbel(gumbel_stream(cfg.cfg_id, layer, step), T * cfg.E).reshape(T, cfg.E)
        return (np.log(p)[None, :] + g).astype(np.float32)
    if cfg.routing == "stream":
        return cache_stream_logits(cfg, layer, step + 1)[step][None, :]
    return normal_f32(logit_stream(cfg.cfg_id, layer, step), T * cfg.E, 1.0).reshape(T, cfg.E)


def cache_stream_sets(cfg: MoEConfig, layer: int, steps: int) -> list:
    """Expert sets of the cache decode stream (batch 1) for steps 0..steps-1.

    Each of the previous token's k experts is kept with probability ``share``;
    the rest are drawn by Gumbel-top-k under Zipf popularity from the experts
    the previous token did not use.
    """
    p = zipf_popularity(cfg, layer)
    logp = np.log(p)
    sets = []
    prev: list = []
    for s in range(steps):
        keep = []
        if prev:
            u = uniform(cache_stream(cfg.cfg_id, layer, s, 0), cfg.k)
            keep = [e for j, e in enumerate(sorted(prev)) if u[j] < cfg.share]
        need = cfg.k - len(keep)
        g = gumbel(cache_stream(cfg.cfg_id, layer, s, 1), cfg.E)
        score = logp + g
        excluded = set(prev)
        cand = [e for e in np.argsort(-score, kind="stable") if int(e) not in excluded]
        chosen = sorted(keep + [int(e) for e in cand[:need]])
        sets.append(chosen)
        prev = chosen
    return sets


def cache_stream_logits(cfg: MoEConfig, layer: int, steps: int) -> np.ndarray:
    """fp32 logits [steps, E] whose top-k is exactly the cache-stream set of each step.

    Chosen experts get 5 + U(0,1); the others min(N(0,1), 3) < 5.
    """
    sets = cache_stream_sets(cfg, layer, steps)
    out = np.empty((steps, cfg.E), dtype=np.float32)
    for s, chosen in enumerate(sets):
        base = np.minimum(normal_f64(cache_stream(cfg.cfg_id, layer, s, 2), cfg.E), 3.0)
        u = uniform(cache_stream(cfg.cfg_id, layer, s, 3), cfg.E)
        base[chosen] = 5.0 + u[chosen]
        out[s] = base.astype(np.float32)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)
