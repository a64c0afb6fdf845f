"""Shared test helpers: parity metrics and oracle-side expert weights."""
from __future__ import annotations

import functools

import numpy as np

import oracle as O
import workloads as W

# acceptance bound on each (step, layer) output
REL_L2_MAX = 5e-3
MAX_ERR_RMS = 2e-2
# routing weights: fp32 expf/sum on the device against fp64 in the oracle
W_REL = 1e-5


def parity_metrics(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(d) / nref if nref > 0 else np.linalg.norm(d)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    maxerr = np.abs(d).max() if d.size else 0.0
    return rel, maxerr, rms


def assert_layer_close(got, ref, what=""):
    rel, maxerr, rms = parity_metrics(got, ref)
    assert rel <= REL_L2_MAX, f"{what}: relative L2 {rel:.3e} > {REL_L2_MAX}"
    assert maxerr <= MAX_ERR_RMS * rms, f"{what}: max |err| {maxerr:.3e} > {MAX_ERR_RMS} * RMS {rms:.3e}"
    return rel, maxerr / rms if rms else 0.0


@functools.lru_cache(maxsize=64)
def oracle_expert(cfg: W.MoEConfig, layer: int, e: int) -> O.QuantizedExpert:
    """The oracle's own quantisation of the generator's fp32 weights for (layer, expert)."""
    return O.QuantizedExpert.from_fp32(*(W.weights_fp32(cfg, layer, e, p) for p in range(3)))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def oracle_expert_from_rows(rows, e: int) -> O.QuantizedExpert:
    """Expert e as the oracle reads it: the device's own row-layout NVFP4 bytes (gate and up are the even and odd
    rows of the interleaved gate/up matrix) and tensor scales, copied to the host."""
    gc = rows.gu_codes[e].cpu().numpy()
    gs = rows.gu_scales[e].cpu().numpy()
    dc = rows.d_codes[e].cpu().numpy()
    ds = rows.d_scales[e].cpu().numpy()
    ts = rows.tscale[e].cpu().numpy()
    return O.QuantizedExpert((np.ascontiguousarray(gc[0::2]), np.ascontiguousarray(gs[0::2]), float(ts[0])),
                             (np.ascontiguousarray(gc[1::2]), np.ascontiguousarray(gs[1::2]), float(ts[1])),
                             (dc, ds, float(ts[2])))


class OracleExperts:
    """expert(e) for O.moe_layer from device row-layout bytes; kept in memory only for small experts."""

    def __init__(self, rows, cache: bool | None = None):
        self.rows = rows
        self.cache = (rows.H * rows.I <= 65536) if cache is None else cache
        self.memo = {}

    def __call__(self, e: int) -> O.QuantizedExpert:
        if not self.cache:
            return oracle_expert_from_rows(self.rows, e)
        if e not in self.memo:
            self.memo[e] = oracle_expert_from_rows(self.rows, e)
        return self.memo[e]
