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
    """Oracle y [L, H] and final state [S, H] for each sampled (b, h).

    The sampled sequences are gathered (on the inputs' device, then copied to
    the host) into one problem of batch 1 whose heads are the pairs, each its
    own group, and the oracle runs once over all of them on every host core."""
    nh = inp["x"].shape[2]
    r = nh // inp["B"].shape[2]
    bi = torch.tensor([b for b, _ in pairs], device=inp["x"].device)
    hi = torch.tensor([h for _, h in pairs], device=inp["x"].device)
    gi = hi // r
    cpu = lambda t: t.detach().cpu()  # noqa: E731
    sub = {
        "x": cpu(inp["x"][bi, :, hi].permute(1, 0, 2).unsqueeze(0)),
        "dt": cpu(inp["dt"][bi, :, hi].permute(1, 0).unsqueeze(0)),
        "A": cpu(inp["A"][hi]),
        "B": cpu(inp["B"][bi, :, gi].permute(1, 0, 2).unsqueeze(0)),
        "C": cpu(inp["C"][bi, :, gi].permute(1, 0, 2).unsqueeze(0)),
        "D": None if inp.get("D") is None else cpu(inp["D"][hi]),
        "initial_state": None if inp.get("initial_state") is None else cpu(inp["initial_state"][bi, hi].unsqueeze(0)),
    }
    res = oracle.ssd_recurrence(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], D=sub["D"],
                                init=sub["initial_state"])
    return {p: (res["y"][0, :, i], res["final_state"][0, i]) for i, p in enumerate(pairs)}


class Guarded:
    """A device tensor with guard regions (canaries) on both sides.

    The whole buffer is filled with a byte pattern; ``t`` is the 4096-byte
    aligned middle part handed to the library as an output, and ``intact()``
    tells whether the guard bytes before and after it are unchanged, i.e.
    whether the kernels wrote only inside the tensor."""
    GUARD = 4096
    PATTERN = 0xA5

    def __init__(self, shape, dtype, device="cuda"):
        elt = torch.empty((), dtype=dtype).element_size()
        n = 1
        for d in shape:
            n *= int(d)
        nbytes = n * elt
        self.buf = torch.full((self.GUARD + nbytes + self.GUARD,), self.PATTERN, dtype=torch.uint8,
                              device=device)
        self.n = nbytes
        self.t = self.buf[self.GUARD:self.GUARD + nbytes].view(dtype).view(*shape)

    def intact(self) -> bool:
        head = self.buf[:self.GUARD]
        tail = self.buf[self.GUARD + self.n:]
        return bool((head == self.PATTERN).all()) and bool((tail == self.PATTERN).all())


# Decay rates for strong-decay tests, cycled over the heads (see
# strong_decay): mild, mixed, mild, mostly direct, mixed, direct.
STRONG_A = (-2.0, -60.0, -8.0, -400.0, -25.0, -1200.0)


def strong_decay(inp: dict, rates=STRONG_A) -> dict:
    """The same inputs with per-head decay rates A[h] = rates[h % len(rates)]
    (an input recipe only: A is a plain input of the layer)."""
    out = dict(inp)
    nh = inp["A"].shape[0]
    out["A"] = torch.tensor([rates[h % len(rates)] for h in range(nh)], dtype=torch.float32,
                            device=inp["A"].device)
    return out


def sample_pairs(batch, nheads, n, seed=0):
    rng = np.random.default_rng(seed)
    all_pairs = [(b, h) for b in range(batch) for h in range(nheads)]
    # always include the first and last pair (index extremes), then random ones
    pick = {0, len(all_pairs) - 1}
    while len(pick) < min(n, len(all_pairs)):
        pick.add(int(rng.integers(len(all_pairs))))
    return [all_pairs[i] for i in sorted(pick)]
