"""Seeded synthetic inputs for the FP8 MoE expert FFN.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It holds no part of the method's arithmetic: it only draws
activations, router logits, expert weights and output gradients with a seeded
torch generator, and turns router logits into (expert id, weight) pairs, which
are inputs of the expert FFN, not steps of it.

Workload shapes follow the five MoE-layer shapes the FFN is measured on
(tokens T, model width D, experts E, top-k, expert hidden width F).  Value
distributions: activations N(0, 1), expert weights N(0, 0.02), output
gradients N(0, 1), router logits N(0, 1) or U(0, 1), or a Zipf(1.2) expert
popularity with Gumbel noise and eight never-routed experts.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

# Scale-mode codes shared by every layer (the C header defines the same
# numbers; they are labels, not arithmetic).
PER_ROW = 0           # one fp32 scale per row
PER_ROW_BLOCK128 = 1  # one fp32 scale per row and per 128 columns
PER_TENSOR = 2        # one fixed fp32 scale for the whole tensor
PER_GROUP_COL = 3     # one fp32 scale per (expert, column) (weight-gradient operands)
MX32 = 4              # MXFP8: one E8M0 (power-of-two) code per row and per 32 columns


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    D: int          # d_model
    E: int          # experts
    k: int          # top-k
    F: int          # d_ff (per expert)
    act_mode: int   # activation (x and h) scale mode
    w_mode: int     # weight scale mode: PER_ROW = per channel, PER_ROW_BLOCK128 = blockwise
    routing: str    # "normal", "uniform" or "zipf"
    backward: bool = False
    w_int8: bool = False  # weight codes int8 instead of e4m3 (activations stay e4m3)

    @property
    def R(self) -> int:
        return self.T * self.k


CONFIGS = {
    "tiny": MoEConfig("tiny", 256, 128, 4, 2, 256, PER_ROW, PER_ROW, "normal"),
    "mixtral": MoEConfig("mixtral", 8192, 4096, 8, 2, 14336, PER_ROW, PER_ROW, "uniform"),
    "dsv3": MoEConfig("dsv3", 16384, 7168, 256, 8, 2048, PER_ROW_BLOCK128,
                      PER_ROW_BLOCK128, "normal"),
    "prefill": MoEConfig("prefill", 2048, 2048, 128, 8, 768, PER_ROW, PER_ROW_BLOCK128, "normal"),
    "fwdbwd": MoEConfig("fwdbwd", 8192, 4096, 64, 6, 1408, PER_TENSOR, PER_TENSOR, "zipf",
                        backward=True),
    # the MXFP8 variant of two of the shapes above (activations, h and
    # weights all in MXFP8)
    "dsv3_mx": MoEConfig("dsv3_mx", 16384, 7168, 256, 8, 2048, MX32, MX32, "normal"),
    "mixtral_mx": MoEConfig("mixtral_mx", 8192, 4096, 8, 2, 14336, MX32, MX32, "uniform"),
    # int8 weights (per channel; blockwise for the prefill chunk) with e4m3
    # activations and h, on two of the shapes above
    "mixtral_w8": MoEConfig("mixtral_w8", 8192, 4096, 8, 2, 14336, PER_ROW, PER_ROW, "uniform", w_int8=True),
    "prefill_w8": MoEConfig("prefill_w8", 2048, 2048, 128, 8, 768, PER_ROW, PER_ROW_BLOCK128, "normal",
                            w_int8=True),
}


def scaled(cfg: MoEConfig, **kw) -> MoEConfig:
    """A copy of `cfg` with some sizes replaced (used for small parity cases)."""
    return dataclasses.replace(cfg, **kw)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def activations(cfg: MoEConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    """x: [T, D] bf16, N(0, 1)."""
    g = _gen(seed * 7919 + 1, device)
    return torch.randn(cfg.T, cfg.D, generator=g, device=device).to(torch.bfloat16)


def output_grad(cfg: MoEConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    """dY: [T, D] bf16, N(0, 1)."""
    g = _gen(seed * 7919 + 5, device)
    return torch.randn(cfg.T, cfg.D, generator=g, device=device).to(torch.bfloat16)


def expert_weights(cfg: MoEConfig, seed: int = 0, device="cpu", std: float = 0.02, experts=None):
    """Expert weights in the device layout, bf16, N(0, std).

    w_in:  [E, 2F, D]  rows 0..F-1 are wi_0, rows F..2F-1 are wi_1 (output
           channel major, the contracted model dimension D contiguous).
    w_out: [E, D, F]   wo, output channel major, F contiguous.

    Every expert draws from generators of its own, so `experts` (a list of
    expert ids) yields exactly those experts' rows of the full tensors,
    without drawing the others."""
    ids = range(cfg.E) if experts is None else list(experts)
    w_in = torch.empty(len(ids), 2 * cfg.F, cfg.D, dtype=torch.bfloat16, device=device)
    w_out = torch.empty(len(ids), cfg.D, cfg.F, dtype=torch.bfloat16, device=device)
    base = (seed * 7919 + 2) * 4099
    for i, e in enumerate(ids):
        g = _gen(base + 2 * e, device)
        w_in[i] = (torch.randn(2 * cfg.F, cfg.D, generator=g, device=device) * std).to(torch.bfloat16)
        g = _gen(base + 2 * e + 1, device)
        w_out[i] = (torch.randn(cfg.D, cfg.F, generator=g, device=device) * std).to(torch.bfloat16)
    return w_in, w_out


def router_logits(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    """[T, E] float64 router logits on the host."""
    g = _gen(seed * 7919 + 3)
    if cfg.routing == "normal":
        return torch.randn(cfg.T, cfg.E, generator=g, dtype=torch.float64).numpy()
    if cfg.routing == "uniform":
        return torch.rand(cfg.T, cfg.E, generator=g, dtype=torch.float64).numpy()
    if cfg.routing == "zipf":
        # Expert popularity: a seeded permutation assigns ranks 1..E; the
        # logit of rank r is -1.2 ln r, plus per-token Gumbel noise, so that
        # taking the top k of the noisy logits samples k experts without
        # replacement in proportion to r^-1.2.  The eight lowest-ranked
        # experts are never routed to.
        rank = torch.randperm(cfg.E, generator=g).numpy() + 1
        base = -1.2 * np.log(rank.astype(np.float64))
        u = torch.rand(cfg.T, cfg.E, generator=g, dtype=torch.float64).numpy()
        u = np.clip(u, 1e-300, 1.0 - 1e-16)
        logits = base[None, :] - np.log(-np.log(u))
        n_masked = min(8, cfg.E - cfg.k)
        masked = rank > cfg.E - n_masked
        logits[:, masked] = -np.inf
        return logits
    raise ValueError(cfg.routing)


def route(logits: np.ndarray, k: int):
    """Softmax over all experts, then the k most probable experts per token.

    Ties go to the lower expert index.  The weights are the selected
    probabilities, not renormalised.  Returns (topk_ids int32 [T, k],
    topk_w float32 [T, k]).
    """
    m = np.max(logits, axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= np.sum(p, axis=1, keepdims=True)
    # stable argsort of -p keeps the lower index first among equal values
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    ids = order.astype(np.int32)
    w = np.take_along_axis(p, order, axis=1).astype(np.float32)
    return ids, w


def routing(cfg: MoEConfig, seed: int = 0):
    return route(router_logits(cfg, seed), cfg.k)


def calibration_scales(cfg: MoEConfig, seed: int = 0) -> dict:
    """Fixed per-tensor scales for the static scheme.

    Each scale is the absolute maximum of an independent calibration draw
    (seed + 1) of the same distribution, divided by 448 (the largest finite
    e4m3 value), frozen afterwards.  h is calibrated from the closed-form
    bound of its distribution rather than a forward pass, which keeps this
    module free of the method's arithmetic: |silu(a0) a1| with a0, a1 of
    standard deviation sigma_a = 0.02 sqrt(D) rarely exceeds (6 sigma_a)^2.
    """
    g = _gen((seed + 1) * 7919 + 11)
    n = min(cfg.T * cfg.D, 1 << 22)
    x_amax = float(torch.randn(n, generator=g).to(torch.bfloat16).float().abs().max())
    nw = min(cfg.F * cfg.D, 1 << 22)
    w0 = float((torch.randn(nw, generator=g) * 0.02).to(torch.bfloat16).float().abs().max())
    w1 = float((torch.randn(nw, generator=g) * 0.02).to(torch.bfloat16).float().abs().max())
    wo = float((torch.randn(nw, generator=g) * 0.02).to(torch.bfloat16).float().abs().max())
    sigma_a = 0.02 * math.sqrt(cfg.D)
    h_amax = (6.0 * sigma_a) ** 2
    f32 = lambda v: float(np.float32(np.float32(v) / np.float32(448.0)))
    return {"x": f32(x_amax), "h": f32(h_amax), "w0": f32(w0), "w1": f32(w1), "wo": f32(wo)}
