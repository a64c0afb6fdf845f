"""The pins of the oracle's Python parts (the slot-cache policy, the MX formats) catch plausible mistakes in them.

Each case builds an altered copy of oracle/lru.py or oracle/mx.py from its source text with one planted mistake,
puts it in place of the original in the pin module, and runs every pin there: at least one must fail.
"""
import importlib
import inspect
import itertools
import os
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

LRU_MUTATIONS = [
    ("evicts the newest", "s = min(cands, key=lambda q: (self.stamp[q], q))",
     "s = min(cands, key=lambda q: (-self.stamp[q], q))"),
    ("eviction ties to the higher slot", "s = min(cands, key=lambda q: (self.stamp[q], q))",
     "s = min(cands, key=lambda q: (self.stamp[q], -q))"),
    ("takes the highest free slot", "            if free:\n                s = free[0]\n            else:\n                cands",
     "            if free:\n                s = free[-1]\n            else:\n                cands"),
    ("hit keeps the old stamp", "                self.stamp[s] = step\n                if self.fetched[s]:",
     "                if self.fetched[s]:"),
    ("prefetch may displace this step's experts", "if self.stamp[s] < step and self.expert_of[s] not in want]",
     "if self.expert_of[s] not in want]"),
    ("prefetch displaces predicted experts", "if self.stamp[s] < step and self.expert_of[s] not in want]",
     "if self.stamp[s] < step]"),
    ("prefetch stamps like a use", "self.stamp[s] = step - 1", "self.stamp[s] = step"),
    ("prefetch refreshes resident experts", "            if e in self.slot_of:\n                continue",
     "            if e in self.slot_of:\n                self.stamp[self.slot_of[e]] = step\n                continue"),
    ("used predictions not counted", "self.prefetch_used += 1", "pass"),
    ("ids visited in the given order", "for e in sorted(ids):", "for e in ids:"),
    ("may evict the token's own experts", "if self.expert_of[s] not in current]", "]"),
    ("resize keeps the oldest", "key=lambda q: (-self.stamp[q], q)", "key=lambda q: (self.stamp[q], q)"),
    ("resize survivors unordered", "resident = sorted(newest_first[:slots])", "resident = newest_first[:slots]"),
    ("resize drops the stamps", "self.stamp = [self.stamp[q] if q >= 0 else -1 for q in moves]",
     "self.stamp = [-1 for q in moves]"),
]

MX_MUTATIONS = [
    ("E2M1 emax off by one", "E2M1_EMAX = 2", "E2M1_EMAX = 3"),
    ("E4M3 emax off by one", "E4M3_EMAX = 8", "E4M3_EMAX = 7"),
    ("ties to the odd code", "(hi % 2 == 0)", "(hi % 2 == 1)"),
    ("exponent not clamped", "return np.clip(x, -127, 127).astype(np.int64)", "return x.astype(np.int64)"),
    ("scale byte bias 126", "scales = (x + 127).astype(np.uint8)", "scales = (x + 126).astype(np.uint8)"),
    ("floor(log2) off by one", "x = np.where(amax > 0, e - 1 - emax, -127)", "x = np.where(amax > 0, e - emax, -127)"),
    ("nibbles swapped", "code = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)",
     "code = ((code[:, 0::2] << 4) | code[:, 1::2]).astype(np.uint8)"),
    ("negative zero kept", "neg = (blocks < 0) & (mag > 0)", "neg = (blocks < 0)"),
    ("E4M3 subnormal step", "m * 2.0 ** -9 if e == 0", "m * 2.0 ** -10 if e == 0"),
]


def mutant_module(path, name, old, new):
    src = open(os.path.join(ROOT, path)).read()
    assert src.count(old) == 1, (name, old)
    mod = types.ModuleType(f"mutant_{name.replace(' ', '_')}")
    mod.__file__ = os.path.join(ROOT, path)
    exec(compile(src.replace(old, new), mod.__file__, "exec"), mod.__dict__)
    return mod


def run_pins(test_mod, params):
    """Runs every test function of test_mod (each parameter set of the parametrised ones); returns the failures."""
    failures = []
    for fname, fn in inspect.getmembers(test_mod, inspect.isfunction):
        if not fname.startswith("test_") or fn.__module__ != test_mod.__name__:
            continue
        for kwargs in params.get(fname, [{}]):
            try:
                fn(**kwargs)
            except Exception as e:  # an assertion or any error the planted mistake causes
                failures.append((fname, kwargs, type(e).__name__))
    return failures


def param_sets(*pairs):
    names = [p[0] for p in pairs]
    return [dict(zip(names, vals)) for vals in itertools.product(*[p[1] for p in pairs])]


@pytest.mark.parametrize("name,old,new", LRU_MUTATIONS, ids=[m[0] for m in LRU_MUTATIONS])
def test_lru_pins_catch(name, old, new, monkeypatch):
    pins = importlib.import_module("test_oracle_lru")
    assert not run_pins(pins, {})   # the original passes
    mut = mutant_module("oracle/lru.py", name, old, new)
    monkeypatch.setattr(pins, "LayerLRU", mut.LayerLRU)
    assert run_pins(pins, {}), f"no pin caught: {name}"


@pytest.mark.parametrize("name,old,new", MX_MUTATIONS, ids=[m[0] for m in MX_MUTATIONS])
def test_mx_pins_catch(name, old, new, monkeypatch):
    pins = importlib.import_module("test_oracle_mx")
    params = {
        "test_block_exponent_on_worked_values": [dict(fmt="mxfp4", emax=2, top=6.0),
                                                 dict(fmt="mxfp8", emax=8, top=448.0)],
        "test_values_on_the_grid_round_trip": param_sets(("fmt", ["mxfp4", "mxfp8"])),
        "test_error_bound_from_the_grid": [dict(fmt="mxfp4", half_step=2.0), dict(fmt="mxfp8", half_step=64.0)],
    }
    # parametrised over the module's own grids: resolved at call time from the module in place
    params["test_rounding_equals_brute_force_nearest"] = [dict(grid=None), dict(grid="e4m3")]
    orig = pins.test_rounding_equals_brute_force_nearest

    def rounding(grid):
        return orig(pins.mx.E2M1_MAG if grid is None else pins.mx.E4M3_MAG)

    monkeypatch.setattr(pins, "test_rounding_equals_brute_force_nearest", rounding)
    rounding.__module__ = pins.__name__
    assert not run_pins(pins, params)   # the original passes
    mut = mutant_module("oracle/mx.py", name, old, new)
    monkeypatch.setattr(pins, "mx", mut)
    assert run_pins(pins, params), f"no pin caught: {name}"
