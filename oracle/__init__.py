"""CPU oracle of the sparse-MoE layer step (fp64, plain C in ``ftoracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the CUDA library never does, and shares no code with
it.  Each step follows the passage cited in ``ftoracle.c``:

* route: softmax over the router logits, top-k (ties to the lower expert
  index), weights renormalised over the selected experts -- page
  "FreeToken：753B大模型塞进单卡的本地部署硬件账该怎么算", MoE core mechanism;
* permute: stable counting sort of (token, slot) pairs by expert;
* expert FFN: SwiGLU over NVFP4 weights dequantised to fp64, h rounded to
  bf16 (mode 0), or with NVFP4 activations as the block-scaled tensor-core
  path computes (mode 1);
* combine: routing-weighted sum in fp64 in slot order, rounded to bf16.

Parity pins live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ftoracle.c")
_LIB = os.path.join(_HERE, "libftoracle.so")
_lock = threading.Lock()
_lib = None

MODE_A16 = 0   # bf16 activations
MODE_A4 = 1    # NVFP4 activations (unit tensor scale)


def build(force: bool = False) -> str:
    """Compile ftoracle.c into oracle/libftoracle.so: gcc -O2, no FMA contraction, OpenMP over rows."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            # FT_ORACLE_LIB: a library built from a deliberately altered copy of ftoracle.c, loaded by the
            # mutation test to check that the pins catch the alteration
            L = ctypes.CDLL(os.environ.get("FT_ORACLE_LIB") or build())
            vp, i64, i32, dbl, flt, u8 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_float, ctypes.c_uint8)
            L.ora_e2m1_value.argtypes, L.ora_e2m1_value.restype = [u8], dbl
            L.ora_e4m3_value.argtypes, L.ora_e4m3_value.restype = [u8], dbl
            L.ora_e2m1_encode.argtypes, L.ora_e2m1_encode.restype = [flt], u8
            L.ora_e4m3_encode.argtypes, L.ora_e4m3_encode.restype = [flt], u8
            L.ora_bf16_round.argtypes, L.ora_bf16_round.restype = [dbl], dbl
            L.ora_quantize_weight.argtypes = [vp, i64, i64, vp, vp, vp]
            L.ora_quantize_act.argtypes = [vp, i64, i64, vp, vp]
            L.ora_dequantize.argtypes = [vp, vp, dbl, i64, i64, vp]
            L.ora_route.argtypes = [vp, i32, i32, i32, vp, vp]
            L.ora_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp]
            L.ora_expert_ffn.argtypes = [vp, vp, vp, i64, i64, vp, i64, i32, vp, vp]
            L.ora_combine.argtypes = [vp, vp, vp, i32, i32, i64, vp, vp]
            L.ora_set_threads.argtypes = [i32]
            L.ora_max_threads.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


class OracleError(ValueError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"oracle {what}: invalid argument")


def set_threads(n: int) -> None:
    lib().ora_set_threads(int(n))


# ---------------------------------------------------------------- formats

def e2m1_value(code: int) -> float:
    return lib().ora_e2m1_value(code)


def e4m3_value(b: int) -> float:
    return lib().ora_e4m3_value(b)


def e2m1_encode(v: float) -> int:
    return lib().ora_e2m1_encode(v)


def e4m3_encode(r: float) -> int:
    return lib().ora_e4m3_encode(r)


def bf16_round(v: float) -> float:
    return lib().ora_bf16_round(v)


def bf16_round_array(a: np.ndarray) -> np.ndarray:
    f = lib().ora_bf16_round
    return np.array([f(float(v)) for v in np.ravel(a)], dtype=np.float64).reshape(np.shape(a))


# ---------------------------------------------------------------- quantisers

def quantize_weight(w: np.ndarray):
    """fp32 [N, K] -> (codes u8 [N, K/2], scales u8 [N, K/16], tensor_scale float)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.empty((N, K // 2), np.uint8)
    scales = np.empty((N, K // 16), np.uint8)
    ts = np.zeros(1, np.float32)
    _check(lib().ora_quantize_weight(_p(w), N, K, _p(codes), _p(scales), _p(ts)), "quantize_weight")
    return codes, scales, float(ts[0])


def quantize_act(x: np.ndarray):
    """fp32 [T, K] -> (codes u8 [T, K/2], scales u8 [T, K/16]) with unit tensor scale."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, K = x.shape
    codes = np.empty((T, K // 2), np.uint8)
    scales = np.empty((T, K // 16), np.uint8)
    _check(lib().ora_quantize_act(_p(x), T, K, _p(codes), _p(scales)), "quantize_act")
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    N = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((N, K), np.float64)
    _check(lib().ora_dequantize(_p(codes), _p(scales), float(tensor_scale), N, K, _p(out)), "dequantize")
    return out


# ---------------------------------------------------------------- layer steps

def route(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(lib().ora_route(_p(logits), T, E, k, _p(ids), _p(w)), "route")
    return ids, w


def permute(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    _check(lib().ora_permute(_p(ids), T, E, k, _p(offsets), _p(perm), _p(inv)), "permute")
    return offsets, perm, inv


def expert_ffn(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, x: np.ndarray, mode: int = MODE_A16):
    """Dequantised fp64 weights, x fp64 [R, H] -> (h [R, I] after bf16 rounding, y [R, H])."""
    Wg, Wu, Wd = (np.ascontiguousarray(a, np.float64) for a in (Wg, Wu, Wd))
    x = np.ascontiguousarray(x, np.float64)
    I, H = Wg.shape
    R = x.shape[0]
    h = np.empty((R, I), np.float64)
    y = np.empty((R, H), np.float64)
    _check(lib().ora_expert_ffn(_p(Wg), _p(Wu), _p(Wd), H, I, _p(x), R, mode, _p(h), _p(y)), "expert_ffn")
    return h, y


def combine(y: np.ndarray, inv: np.ndarray, w: np.ndarray, T: int, k: int):
    y = np.ascontiguousarray(y, np.float64)
    inv = np.ascontiguousarray(inv, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    H = y.shape[1]
    out = np.empty((T, H), np.float64)
    pre = np.empty((T, H), np.float64)
    _check(lib().ora_combine(_p(y), _p(inv), _p(w), T, k, H, _p(out), _p(pre)), "combine")
    return out, pre


class QuantizedExpert:
    """One expert's three NVFP4 tensors as the oracle quantised them, plus their fp64 dequantisation."""

    def __init__(self, gate, up, down):
        self.q = (gate, up, down)   # each (codes, scales, tensor_scale)
        self.Wg, self.Wu, self.Wd = (dequantize(*t) for t in self.q)

    @classmethod
    def from_fp32(cls, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> "QuantizedExpert":
        return cls(quantize_weight(wg), quantize_weight(wu), quantize_weight(wd))


def moe_layer(logits: np.ndarray, x_bf16_bits: np.ndarray, k: int, expert, mode: int = MODE_A16,
              rows: np.ndarray | None = None):
    """Full layer step: route -> permute -> expert FFN -> combine.

    ``expert(e)`` returns a QuantizedExpert.  ``rows`` (optional) restricts the
    FFN and the combine to those tokens (route and permute still cover all).
    Returns a dict with ids, w, offsets, perm, inv, h, y (per permuted row,
    NaN where not computed), out (bf16 values as fp64, [len(rows), H]).
    """
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    x = (np.ascontiguousarray(x_bf16_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    H = x.shape[1]
    ids, w = route(logits, k)
    offsets, perm, inv = permute(ids, E)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    need = np.zeros(T * k, bool)
    for t in rows:
        need[inv[t * k:(t + 1) * k]] = True
    y = np.full((T * k, H), np.nan)
    h = None
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        ps = [p for p in range(lo, hi) if need[p]]
        if not ps:
            continue
        ex = expert(e)
        toks = perm[ps] // k
        he, ye = expert_ffn(ex.Wg, ex.Wu, ex.Wd, x[toks], mode)
        if h is None:
            h = np.full((T * k, he.shape[1]), np.nan)
        h[ps] = he
        y[ps] = ye
    sub_inv = inv.reshape(T, k)[rows].reshape(-1)
    out, pre = combine(y, sub_inv, w[rows], len(rows), k)
    return dict(ids=ids, w=w, offsets=offsets, perm=perm, inv=inv, h=h, y=y, out=out, out_pre=pre, rows=rows)
