"""Helpers for the GPU parity tests: device transfer, oracle on sampled
(batch, head) pairs, and the error metric.  The oracle is fed only the
seeded inputs (or its own intermediate results), never a CUDA output."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances on max|err| / max|ref|: 2e-2 with bf16 operands and fp32
# accumulation, 1e-4 on the fp32 path.
TOL = {"bf16": 2e-2, "fp32": 1e-4}


def rel_err(a, ref) -> float:
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(a - ref))) / max(den, 1e-30)


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device).contiguous() if v is not None else None) for k, v in inp.items()}


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def pair_problem(inp: dict, b: int, heads) -> dict:
    """The sub-problem of batch row b and the listed heads, each head given its
    own group (an exact re-expression: a head only ever reads its group)."""
    nh = inp["x"].shape[2]
    G = inp["B"].shape[2]
    r = nh // G
    heads = list(heads)
    groups = [h // r for h in heads]
    sub = {
        "x": inp["x"][b:b + 1, :, heads],
        "dt": inp["dt"][b:b + 1, :, heads],
        "A": inp["A"][heads],
        "B": inp["B"][b:b + 1, :, groups],
        "C": inp["C"][b:b + 1, :, groups],
        "D": None if inp.get("D") is None else inp["D"][heads],
        "initial_state": None if inp.get("initial_state") is None else inp["initial_state"][b:b + 1, heads],
    }
    return sub


def oracle_pairs(inp: dict, pairs) -> dict:
    """Oracle y [L, H] and final state [S, H] for each sampled (b, h)."""
    by_b = {}
    for b, h in pairs:
        by_b.setdefault(b, []).append(h)
    out = {}
    for b, heads in by_b.items():
        sub = pair_problem(inp, b, heads)
        r = oracle.ssd_recurrence(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], D=sub["D"],
                                  init=sub["initial_state"])
        for i, h in enumerate(heads):
            out[(b, h)] = (r["y"][0, :, i], r["final_state"][0, i])
    return out


def sample_pairs(batch, nheads, n, seed=0):
    rng = np.random.default_rng(seed)
    all_pairs = [(b, h) for b in range(batch) for h in range(nheads)]
    # always include the first and last pair (index extremes), then random ones
    pick = {0, len(all_pairs) - 1}
    while len(pick) < min(n, len(all_pairs)):
        pick.add(int(rng.integers(len(all_pairs))))
    return [all_pairs[i] for i in sorted(pick)]
