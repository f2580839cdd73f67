"""Independent pins for the fp64 oracle.

Each function here computes something the blog or plain mathematics fixes
WITHOUT going through the oracle's own formula, then reports how far the
oracle is from it.  Source: "Accelerating Mamba-2 with High-Performance Forward
Pass Kernels in NVIDIA CUDA Tile" (NVIDIA technical blog), cited as
[blog §section].  Used by test_oracle_pins.py and, against deliberately broken
copies of the oracle, by test_oracle_mutants.py.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_err(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = max(float(np.max(np.abs(ref))) if ref.size else 0.0, 1e-300)
    return float(np.max(np.abs(a - ref))) / den if ref.size else 0.0


def random_problem(seed, b, L, nh, H, S, G, init=True, a_zero=False, dt_zero=False):
    """fp64 inputs with the decays of a real layer (A < 0, dt > 0)."""
    rng = np.random.default_rng(seed)
    p = {
        "x": rng.standard_normal((b, L, nh, H)),
        "dt": np.zeros((b, L, nh)) if dt_zero else rng.uniform(0.01, 0.6, (b, L, nh)),
        "A": np.zeros(nh) if a_zero else -rng.uniform(0.3, 3.0, nh),
        "B": rng.standard_normal((b, L, G, S)),
        "C": rng.standard_normal((b, L, G, S)),
        "D": rng.standard_normal(nh),
        "init": rng.standard_normal((b, nh, S, H)) if init else None,
    }
    return p


def _group(nh, G, h):
    return h // (nh // G)


# --------------------------------------------------------------- pin 1
def brute_force(p):
    """Unrolled expansion of the recurrence [blog §Mamba-2 architecture, the
    expansion of h_{t+T}]: h_t = exp(sum_{k<=t} a_k) h_0
    + sum_{j<=t} exp(sum_{j<k<=t} a_k) b_j x_j^T, then y_t = C_t^T h_t + D x_t.
    Every exponent is summed afresh (no running product), O(L^2 S H)."""
    x, dt, A, B, C, D, h0 = (p[k] for k in ("x", "dt", "A", "B", "C", "D", "init"))
    b, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    fin = np.zeros((b, nh, S, H))
    for bi in range(b):
        for h in range(nh):
            g = _group(nh, G, h)
            a = A[h] * dt[bi, :, h]
            start = h0[bi, h] if h0 is not None else np.zeros((S, H))
            for t in range(L):
                ht = np.exp(a[: t + 1].sum()) * start
                for j in range(t + 1):
                    ht = ht + np.exp(a[j + 1: t + 1].sum()) * dt[bi, j, h] * np.outer(B[bi, j, g],
                                                                                    x[bi, j, h])
                y[bi, t, h] = C[bi, t, g] @ ht + D[h] * x[bi, t, h]
                if t == L - 1:
                    fin[bi, h] = ht
            if L == 0:
                fin[bi, h] = start
    return y, fin


# --------------------------------------------------------------- pin 2
def linear_attention_closed_form(p):
    """A = 0 removes the decay and the layer is linear attention
    [blog §Mamba-2 architecture, Y = C h + ((C B^T) . M) X + D X]:
    Y = C h_0 + tril(C B^T) (dt . X) + D X, final = h_0 + (dt . B)^T X,
    with the diagonal kept (inclusive causal mask)."""
    x, dt, B, C, D, h0 = (p[k] for k in ("x", "dt", "B", "C", "D", "init"))
    b, L, nh, H = x.shape
    G, S = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    fin = np.zeros((b, nh, S, H))
    for bi in range(b):
        for h in range(nh):
            g = _group(nh, G, h)
            Cm, Bm, X = C[bi, :, g], B[bi, :, g], x[bi, :, h]
            start = h0[bi, h] if h0 is not None else np.zeros((S, H))
            M = np.tril(np.ones((L, L)))
            y[bi, :, h] = Cm @ start + ((Cm @ Bm.T) * M) @ (dt[bi, :, h][:, None] * X) + D[h] * X
            fin[bi, h] = start + (dt[bi, :, h][:, None] * Bm).T @ X
    return y, fin


# --------------------------------------------------------------- pin 8
def geometric_closed_form(L, alpha, delta, beta, gamma, xi, dcoef, h0):
    """Scalar state (S = H = 1) with constant inputs: the recurrence is a
    first-order linear filter, h_t = r^t h_0 + delta*beta*xi (1 - r^t)/(1 - r),
    r = exp(alpha*delta); y_t = gamma h_t + D xi."""
    r = np.exp(alpha * delta)
    t = np.arange(1, L + 1)
    h = r ** t * h0 + delta * beta * xi * (1.0 - r ** t) / (1.0 - r)
    return gamma * h + dcoef * xi, h[-1]


def read_golden(name):
    """Parse one [section] of tests/golden/hand_worked_examples.txt."""
    path = os.path.join(GOLDEN, "hand_worked_examples.txt")
    sect, cur = {}, None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                continue
            if cur == name:
                k, v = line.split(":", 1)
                sect[k.strip()] = np.array([float(s) for s in v.split(",")])
    b, L, nh, H, S, G = (int(v) for v in sect["shape"])
    return {
        "x": sect["x"].reshape(b, L, nh, H), "dt": sect["dt"].reshape(b, L, nh),
        "A": sect["A"].reshape(nh), "D": sect["D"].reshape(nh),
        "B": sect["B"].reshape(b, L, G, S), "C": sect["C"].reshape(b, L, G, S),
        "init": sect["initial_state"].reshape(b, nh, S, H),
        "y": sect["y"].reshape(b, L, nh, H), "final_state": sect["final_state"].reshape(b, nh, S, H),
    }


# --------------------------------------------------------------- suite
def run_suite(oracle):
    """Every pin against the given oracle module; returns {pin: error}.

    Errors are max|diff| / max|ref| (0 for exact checks that pass, 1.0 for
    exact checks that fail)."""
    res = {}
    # pin 1: brute force, several heads, 2 groups, decay on
    p = random_problem(1, 2, 9, 4, 3, 4, 2)
    yb, fb = brute_force(p)
    r = oracle.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"])
    res["brute_force_y"] = rel_err(r["y"], yb)
    res["brute_force_final"] = rel_err(r["final_state"], fb)
    # pin 2: A = 0 closed form, recurrence and chunked
    p = random_problem(2, 2, 13, 2, 3, 5, 1, a_zero=True)
    yc, fc = linear_attention_closed_form(p)
    r = oracle.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"])
    res["a0_recurrence_y"] = rel_err(r["y"], yc)
    res["a0_recurrence_final"] = rel_err(r["final_state"], fc)
    ch = oracle.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"], 4, D=p["D"], init=p["init"])
    res["a0_chunked_y"] = rel_err(ch["y"], yc)
    res["a0_chunked_final"] = rel_err(ch["final_state"], fc)
    # pin 3: dt = 0 keeps the state; y = C h0 + D x
    p = random_problem(3, 1, 10, 2, 3, 4, 1, dt_zero=True)
    for name, run in (("rec", lambda: oracle.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"],
                                                            D=p["D"], init=p["init"])),
                      ("chunked", lambda: oracle.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"],
                                                             4, D=p["D"], init=p["init"]))):
        r = run()
        res[f"dt0_{name}_final"] = 0.0 if np.array_equal(r["final_state"], p["init"]) else 1.0
        yref = np.einsum("blgs,bhsk->blhk", p["C"], p["init"]) + p["D"][None, None, :, None] * p["x"]
        res[f"dt0_{name}_y"] = rel_err(r["y"], yref)
    # pin 4: chunked == sequential at several chunk sizes, including ragged
    p = random_problem(4, 2, 23, 3, 5, 6, 3)
    r = oracle.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"],
                              chunk_size=5)
    worst_y = worst_f = worst_s = 0.0
    for T in (1, 2, 4, 5, 8, 16, 23, 64):
        ch = oracle.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"], T, D=p["D"], init=p["init"])
        worst_y = max(worst_y, rel_err(ch["y"], r["y"]))
        worst_f = max(worst_f, rel_err(ch["final_state"], r["final_state"]))
        if T == 5:
            worst_s = rel_err(ch["chunk_states"], r["chunk_states"])
    res["chunked_vs_rec_y"], res["chunked_vs_rec_final"] = worst_y, worst_f
    res["chunked_vs_rec_chunk_states"] = worst_s
    # pin 5: split sequence, run(L) == run(L1) -> run(L - L1, init = final)
    p = random_problem(5, 1, 24, 2, 3, 4, 1)
    full = oracle.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"], 8, D=p["D"], init=p["init"])
    first = oracle.ssd_chunked(p["x"][:, :16], p["dt"][:, :16], p["A"], p["B"][:, :16],
                               p["C"][:, :16], 8, D=p["D"], init=p["init"])
    second = oracle.ssd_chunked(p["x"][:, 16:], p["dt"][:, 16:], p["A"], p["B"][:, 16:],
                                p["C"][:, 16:], 8, D=p["D"], init=first["final_state"])
    res["split_y"] = rel_err(np.concatenate([first["y"], second["y"]], axis=1), full["y"])
    res["split_final"] = rel_err(second["final_state"], full["final_state"])
    # pin 6: causality, perturbing token t' leaves y_{<t'} bit-identical
    p = random_problem(6, 1, 16, 2, 3, 4, 1)
    base = oracle.ssd_chunked(p["x"], p["dt"], p["A"], p["B"], p["C"], 8, D=p["D"], init=p["init"])
    bad = 0.0
    for tp in (3, 8, 13):
        q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
        q["x"][:, tp] += 1.0
        q["B"][:, tp] -= 2.0
        q["C"][:, tp] *= 3.0
        q["dt"][:, tp] += 0.25
        pert = oracle.ssd_chunked(q["x"], q["dt"], q["A"], q["B"], q["C"], 8, D=q["D"],
                                  init=q["init"])
        if not np.array_equal(pert["y"][:, :tp], base["y"][:, :tp]):
            bad = 1.0
        if np.array_equal(pert["y"][:, tp], base["y"][:, tp]):
            bad = 1.0  # the perturbed token must matter to itself
    res["causality"] = bad
    # pin 7: groups, G = nh equals G = 1 with B, C repeated per head
    p = random_problem(7, 1, 12, 4, 3, 4, 1)
    one = oracle.ssd_recurrence(p["x"], p["dt"], p["A"], p["B"], p["C"], D=p["D"], init=p["init"])
    rep = {k: v for k, v in p.items()}
    rep["B"] = np.repeat(p["B"], 4, axis=2)
    rep["C"] = np.repeat(p["C"], 4, axis=2)
    four = oracle.ssd_recurrence(rep["x"], rep["dt"], rep["A"], rep["B"], rep["C"], D=rep["D"],
                                 init=rep["init"])
    res["groups_repeat"] = 0.0 if np.array_equal(one["y"], four["y"]) else 1.0
    # pin 8: scalar geometric closed form and the hand-worked fixtures
    L, alpha, delta, beta, gamma, xi, dc, h0 = 40, -1.3, 0.2, 0.7, -1.1, 0.9, 0.4, 2.5
    ones = np.ones((1, L, 1, 1))
    r = oracle.ssd_recurrence(xi * ones, delta * np.ones((1, L, 1)), np.array([alpha]),
                              beta * ones, gamma * ones, D=np.array([dc]),
                              init=np.full((1, 1, 1, 1), h0))
    yg, fg = geometric_closed_form(L, alpha, delta, beta, gamma, xi, dc, h0)
    res["geometric_y"] = rel_err(r["y"].reshape(-1), yg)
    res["geometric_final"] = rel_err(r["final_state"].reshape(-1), [fg])
    for name in ("scalar_geometric", "two_by_two"):
        gd = read_golden(name)
        r = oracle.ssd_recurrence(gd["x"], gd["dt"], gd["A"], gd["B"], gd["C"], D=gd["D"],
                                  init=gd["init"])
        ch = oracle.ssd_chunked(gd["x"], gd["dt"], gd["A"], gd["B"], gd["C"], 2, D=gd["D"],
                                init=gd["init"])
        res[f"golden_{name}"] = max(rel_err(r["y"], gd["y"]), rel_err(r["final_state"], gd["final_state"]),
                                    rel_err(ch["y"], gd["y"]),
                                    rel_err(ch["final_state"], gd["final_state"]))
    # pin 9: stage 1 on constant inputs is a linear ramp restarting per chunk
    b, L, nh, T = 2, 21, 3, 8
    dtc = np.full((b, L, nh), 0.125)
    Ac = np.array([-1.0, -2.5, -0.5])
    G = oracle.chunk_cumsum(dtc, Ac, T)
    ramp = (np.arange(L) % T + 1)[None, None, :] * (Ac[None, :, None] * 0.125) / np.log(2.0)
    res["cumsum_ramp"] = rel_err(G, np.broadcast_to(ramp, G.shape))
    return res


# Tolerances for fp64: the pinned quantities differ from the oracle only by
# summation order, so they agree to ~1e-15 relative; 1e-12 leaves room for
# cancellation at these sizes while any real slip (a missing term, a sign, an
# index) moves the error to O(1e-2) or more.
TOL = 1e-12
