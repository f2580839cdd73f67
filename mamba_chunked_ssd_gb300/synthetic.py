"""Seeded synthetic inputs for the Mamba-2 SSD forward pass.

This module draws inputs only; it holds none of the method's arithmetic.  The
CUDA path, the oracle and the benchmark all take their inputs from here, so the
two sides of every comparison see the same rounded values.

Distributions (per workload description):
  x, B, C ~ N(0, 1), rounded to the workload dtype (bf16 or fp32);
  dt = clip(softplus(N(mu, 1)), 1e-3, 0.1) in fp32 (mu = -3, or -4 for the
       long-memory large-state workload);
  A = -exp(U(ln 1, ln 16)) per head, fp32, so A lies in [-16, -1];
  D ~ N(0, 1) per head, fp32;
  initial_state ~ N(0, 0.1) fp32 when the workload carries a state, else None.
Draws come from one ``torch.Generator`` seeded per call, in the fixed order
x, dt, A, B, C, D, initial_state.  By default the generator runs on the CPU
(the same values on every machine); ``device="cuda"`` draws on the GPU instead,
which is much faster for the large sweep shapes (different values for the same
seed, but still one seeded draw that both sides of a comparison share).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    dtype: str = "bf16"          # dtype of x, B, C, y and chunk states
    dt_mu: float = -3.0          # mean of the normal fed to softplus
    init_state: bool = False     # draw a carried initial state
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    @property
    def nchunks(self) -> int:
        return -(-self.seqlen // self.chunk_size)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The named workloads.  Sizes follow the workload descriptions; the first is
# small enough for the fp64 oracle to finish in well under a second.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 256, 2, 16, 16, 1, 64, dtype="fp32"),
    "mamba2_1p3b_layer": Workload("mamba2_1p3b_layer", 2, 2048, 64, 64, 128, 1, 256),
    "long_seq_carried_state": Workload("long_seq_carried_state", 4, 8192, 64, 64, 128, 1, 256,
                                       init_state=True),
    "large_state": Workload("large_state", 2, 16384, 32, 128, 256, 8, 128, dt_mu=-4.0),
    # one decode step (seqlen 1) for 256 sequences of the same layer, each
    # carrying a state: the inference use of the carried final state
    "decode_b256": Workload("decode_b256", 256, 1, 64, 64, 128, 1, 1, init_state=True),
    # the example problem the blog's usage snippet times: batch 4, 16384
    # tokens, one group, 8 heads, state 128, head dim 64, chunk 128
    "blog_example": Workload("blog_example", 4, 16384, 8, 64, 128, 1, 128),
    # the long-sequence layer in fp32 with chunks of 128 (the fp32 path's
    # tensor-core shapes)
    "long_seq_fp32_t128": Workload("long_seq_fp32_t128", 4, 8192, 64, 64, 128, 1, 128, dtype="fp32",
                                   init_state=True),
}


def sweep_workloads(seeds=(0, 1, 2)):
    """The bf16 sweep: batch*L = 65536 tokens, 64 heads, 1 group."""
    out = []
    for L in (1024, 4096, 16384, 32768):
        for S in (64, 128, 256):
            for H in (64, 128):
                for T in (128, 256):
                    for seed in seeds:
                        out.append(Workload(f"sweep_L{L}_S{S}_H{H}_T{T}", 65536 // L, L, 64, H, S,
                                            1, T, seed=seed))
    return out


TORCH_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


def make_inputs(w: Workload, seed: int | None = None, device: str = "cpu") -> dict:
    """Draw the inputs of workload ``w`` on ``device`` (CPU by default).

    Returns a dict of tensors on that device: x [b,L,nh,H], dt [b,L,nh],
    A [nh], B, C [b,L,G,S], D [nh], initial_state [b,nh,S,H] or None."""
    g = torch.Generator(device=device).manual_seed(w.seed if seed is None else seed)
    dt_ = TORCH_DTYPES[w.dtype]
    b, L, nh, H, S, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    kw = {"generator": g, "device": device}
    x = torch.randn(b, L, nh, H, **kw).to(dt_)
    dt = torch.nn.functional.softplus(torch.randn(b, L, nh, **kw) + w.dt_mu)
    dt = dt.clamp_(1e-3, 0.1).float()
    A = -torch.exp(torch.rand(nh, **kw) * math.log(16.0)).float()
    B = torch.randn(b, L, G, S, **kw).to(dt_)
    C = torch.randn(b, L, G, S, **kw).to(dt_)
    D = torch.randn(nh, **kw).float()
    init = (torch.randn(b, nh, S, H, **kw) * 0.1).float() if w.init_state else None
    return {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "initial_state": init}
