"""Seeded synthetic workloads for the routed-expert MoE layer.

This module is the only code shared by the oracle side and the CUDA side of
the tests and the benchmark: it draws inputs (tokens, routing decisions,
weights, output gradients) and holds none of the layer's arithmetic.  The
router that turns logits into top-K IDs and scores belongs to the caller of
the layer, so it lives here as input generation.

Workloads (names used by tests and the benchmark):

* ``tiny_bf16``   T=128, D=256, F=512, E=8, K=2.  Top-2 of N(0,1) logits,
  softmax over the two, 5% of routes inactive.  BF16.
* ``e64_bf16``    T=2048, D=2048, F=1408, E=64, K=6.  Uniform K-of-E
  without repeat, scores = softmax of K N(0,1) draws.  BF16.
* ``e384_mxfp8``  T=2048, D=7168, F=2048, E=384, K=6, uniform routing,
  MXFP8 routed experts plus one BF16 shared expert of F=2048.
* ``e384_mxfp8_zipf_train``  the same shapes, forward + backward, expert
  popularity Zipf(1.2) over a seeded rank->expert permutation, 10% inactive.
* ``ten_layer_graph``  10 MXFP8 layers, T=4096, D=7168, F=2048, E=384,
  K=8, each layer Zipf(s ~ U[0.8, 1.5]) with its own seed.
* ``e6_dense``    diagnostic: the e384 shapes with E=6, K=6, so every
  token visits every expert (2048 rows per expert).
* ``profile_e24`` the e384 per-expert shape with 24 experts and T=128, a
  small case for hardware-counter captures.

Weights are N(0, 1/D) for W13 and N(0, 1/F) for W2, tokens and output
gradients N(0, 1), all rounded to BF16.
"""

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    F: int
    E: int
    K: int
    precision: str            # "bf16", "mxfp8" or "nvfp4" (inference)
    routing: str              # "topk_logits", "uniform", "zipf"
    inactive_frac: float = 0.0
    zipf_s: float = 1.2
    shared_F: int = 0         # 0: no shared expert
    train: bool = False
    layers: int = 1
    seed: int = 0


WORKLOADS = {
    "tiny_bf16": Workload("tiny_bf16", 128, 256, 512, 8, 2, "bf16", "topk_logits",
                          inactive_frac=0.05, train=True, seed=1),
    "e64_bf16": Workload("e64_bf16", 2048, 2048, 1408, 64, 6, "bf16", "uniform", seed=2),
    "e384_mxfp8": Workload("e384_mxfp8", 2048, 7168, 2048, 384, 6, "mxfp8", "uniform",
                           shared_F=2048, seed=3),
    "e384_mxfp8_zipf_train": Workload("e384_mxfp8_zipf_train", 2048, 7168, 2048, 384, 6,
                                      "mxfp8", "zipf", inactive_frac=0.10, zipf_s=1.2,
                                      shared_F=2048, train=True, seed=4),
    "ten_layer_graph": Workload("ten_layer_graph", 4096, 7168, 2048, 384, 8, "mxfp8",
                                "zipf", train=True, layers=10, seed=5),
    "e6_dense": Workload("e6_dense", 2048, 7168, 2048, 6, 6, "mxfp8", "uniform", seed=6),
    # the e384 inference shape's routed layer with NVFP4 experts (inference
    # only; no shared expert)
    "e384_nvfp4": Workload("e384_nvfp4", 2048, 7168, 2048, 384, 6, "nvfp4", "uniform", seed=11),
    # profiling case: the e384 per-expert shape (about 32 rows per expert, D=7168,
    # F=2048) with 24 experts, so a full ncu capture holds a few GB, while the
    # weight gradients (1.4 GB for W13) still exceed L2
    "profile_e24": Workload("profile_e24", 128, 7168, 2048, 24, 6, "mxfp8", "zipf", inactive_frac=0.10,
                            zipf_s=1.2, train=True, seed=7),
    # decode-sized steps (diagnostic): the e384 MXFP8 inference shapes with 1
    # and 16 tokens, no shared expert; only the routed experts' weights stream
    "decode_e384_t1": Workload("decode_e384_t1", 1, 7168, 2048, 384, 6, "mxfp8", "uniform", seed=9),
    "decode_e384_t16": Workload("decode_e384_t16", 16, 7168, 2048, 384, 6, "mxfp8", "uniform", seed=10),
    "decode_e384_t1_nvfp4": Workload("decode_e384_t1_nvfp4", 1, 7168, 2048, 384, 6, "nvfp4", "uniform", seed=9),
    # profiling case for the row-sized kernels (gathers, combine): the e384
    # token count and width (T=2048, D=7168, K=6, so about 12 K routed rows)
    # with 32 experts, about 10 GB on the device
    # profiling case of the NVFP4 GEMMs: the e384 token count and widths with
    # 32 experts (about 3 routing blocks each), about 1 GB of NVFP4 weights
    "profile_e32_nvfp4": Workload("profile_e32_nvfp4", 2048, 7168, 2048, 32, 6, "nvfp4", "uniform", seed=12),
    "profile_e32": Workload("profile_e32", 2048, 7168, 2048, 32, 6, "mxfp8", "zipf", inactive_frac=0.10,
                            zipf_s=1.2, train=True, seed=8),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return replace(w, **kw)


# ------------------------------------------------------------------ routing

def _gumbel_topk(rng, logits, k):
    g = -np.log(-np.log(rng.uniform(1e-12, 1.0, size=logits.shape)))
    return np.argsort(-(logits + g), axis=1, kind="stable")[:, :k]


def make_routing(w: Workload, layer: int = 0, zipf_s=None):
    """Top-K expert IDs [T,K] int32 and scores [T,K] float32 (caller's router)."""
    rng = np.random.default_rng(1000 * w.seed + 17 * layer + 1)
    T, E, K = w.T, w.E, w.K
    if w.routing == "topk_logits":
        logits = rng.standard_normal((T, E))
        ids = np.argsort(-logits, axis=1, kind="stable")[:, :K]
        sel = np.take_along_axis(logits, ids, axis=1)
    else:
        if w.routing == "uniform":
            base = np.zeros((T, E))
        elif w.routing == "zipf":
            s = w.zipf_s if zipf_s is None else zipf_s
            rank_to_expert = rng.permutation(E)
            p = np.empty(E)
            p[rank_to_expert] = 1.0 / np.arange(1, E + 1) ** s
            base = np.broadcast_to(np.log(p / p.sum()), (T, E))
        else:
            raise ValueError(w.routing)
        ids = _gumbel_topk(rng, base, K)
        sel = rng.standard_normal((T, K))
    sel = sel - sel.max(axis=1, keepdims=True)
    scores = np.exp(sel) / np.exp(sel).sum(axis=1, keepdims=True)
    ids = ids.astype(np.int32)
    scores = scores.astype(np.float32)
    n_off = int(round(w.inactive_frac * T * K))
    if n_off:
        off = rng.permutation(T * K)[:n_off]
        ids.reshape(-1)[off] = -1
        scores.reshape(-1)[off] = 0.0
    return ids, scores


def layer_zipf_s(w: Workload, layer: int) -> float:
    """Per-layer skew of the ten-layer workload, s ~ U[0.8, 1.5] (seeded)."""
    return float(np.random.default_rng(w.seed * 7919 + layer).uniform(0.8, 1.5))


# ------------------------------------------------------------------ tensors

def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_tokens(w: Workload, device="cpu", layer: int = 0, salt: int = 0):
    """x [T,D] ~ N(0,1) in BF16."""
    g = _gen(device, 10_000 * w.seed + 31 * layer + salt + 11)
    return torch.randn((w.T, w.D), generator=g, device=device).to(torch.bfloat16)


def make_grad_out(w: Workload, device="cpu", layer: int = 0):
    """dY [T,D] ~ N(0,1) in BF16."""
    return make_tokens(w, device, layer, salt=5)


def make_weights(w: Workload, device="cpu", layer: int = 0, E=None, F=None, experts=None):
    """W13 [E,2F,D] ~ N(0,1/D) and W2 [E,D,F] ~ N(0,1/F), BF16.

    Rows 0..F-1 of W13 are the gate projection, rows F..2F-1 the up
    projection.  Each expert has its own seed, so ``experts`` (a list of
    expert indices) draws exactly those experts' weights of the full set."""
    E = w.E if E is None else E
    F = w.F if F is None else F
    experts = list(range(E)) if experts is None else list(experts)
    n = len(experts)
    w13 = torch.empty((n, 2 * F, w.D), device=device, dtype=torch.bfloat16)
    w2 = torch.empty((n, w.D, F), device=device, dtype=torch.bfloat16)
    g = torch.Generator(device=device)
    for i, e in enumerate(experts):
        g.manual_seed(20_000 * w.seed + 97 * layer + 1_000_003 * (E + 3) + 7919 * e)
        w13[i] = (torch.randn((2 * F, w.D), generator=g, device=device) * w.D ** -0.5).to(torch.bfloat16)
        w2[i] = (torch.randn((w.D, F), generator=g, device=device) * F ** -0.5).to(torch.bfloat16)
    return w13, w2


def make_shared_weights(w: Workload, device="cpu", layer: int = 0):
    """One dense shared expert (E=1, F=shared_F) in BF16."""
    return make_weights(w, device, layer=layer + 500, E=1, F=w.shared_F)
