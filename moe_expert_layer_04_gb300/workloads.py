"""Seeded synthetic inputs for the routed MoE layer.

This module only draws random numbers in the shapes and distributions of the
layer's workloads; it holds none of the layer's arithmetic, so both the CUDA
path and the CPU oracle may take their inputs from it.

Every tensor has its own ``torch.Generator`` seeded from ``(seed, name)``
with a stable hash, so any subset of tensors can be regenerated on its own.
The same call on the same device gives the same bits; CPU and CUDA
generators give different (equally distributed) streams.

Shapes and distributions follow the five workloads the layer is measured on
(DeepSeek-V4.1-Flash MoE layer: 384 routed experts, top-6, one shared expert,
as in "MindSpore HyperParallel一键开箱DeepSeek-V4.1-Flash", §01):

  tiny_fwd          T=64,    d=128,  E=16,  k=2, I=64,   rho=1.0
  full_fwd          T=4096,  d=4096, E=384, k=6, I=2048, rho=2.5, near-uniform load
  skewed_mm_fwd     T=8192,  ... 25% vision tokens, Zipf(1.1) expert load,
                    hash-router variant (tid2eid [129280, 6], input ids Zipf(1.0))
  fwd_bwd           T=8192,  ... upstream gradient dY ~ N(0, 1)
  long_slice_fwd_bwd T=65536, ... 30% vision, Zipf(1.1) load, recompute
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch

VOCAB = 129280
VISION_BLOCK = 576

# Scale of the per-expert logit offsets that skew the expert load towards a
# Zipf(1.1) rank-frequency law: offset[e] = -ZIPF_LAMBDA * s * ln(rank[e]).
# Calibrated once with the oracle's routing on full-width synthetic inputs by
# `python -m oracle.calibrate_zipf` (least-squares slope of log count against log rank
# over ranks 2..384 within 0.05 of -1.1).
ZIPF_LAMBDA = 0.4767


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    rho: float
    clamp: float = 7.0
    vision_frac: float = 0.0
    zipf_s: float = 0.0          # expert-load skew exponent (0 = none)
    hash_variant: bool = False   # also draw tid2eid and Zipf(1.0) input ids
    bias_amp: float = 0.1        # routing bias ~ U(-bias_amp, bias_amp)
    backward: bool = False
    recompute: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def S(self) -> int:
        return self.T * self.k


# The full-width near-uniform workloads draw the routing bias from
# U(-0.01, 0.01): with logits of std 1.28 (x ~ N(0,1), W_g ~ N(0,0.02),
# d = 4096) a selection of 6 of 384 experts sits where a bias of 0.1 is worth
# about 1.4 logit standard deviations, and U(-0.1, 0.1) leaves ~110 of the 384
# experts without a token (the hottest gets ~300 rows), which is not the
# near-uniform ~64 tokens/expert load these workloads stand for.  At 0.01 the
# load is 43..96 rows per expert.  "full_fwd_bias0.1" keeps the literal range.
WORKLOADS = {
    "tiny_fwd": Workload("tiny_fwd", 64, 128, 16, 2, 64, 1.0),
    "full_fwd": Workload("full_fwd", 4096, 4096, 384, 6, 2048, 2.5, bias_amp=0.01),
    "full_fwd_bias0.1": Workload("full_fwd_bias0.1", 4096, 4096, 384, 6, 2048, 2.5),
    "skewed_mm_fwd": Workload("skewed_mm_fwd", 8192, 4096, 384, 6, 2048, 2.5,
                              vision_frac=0.25, zipf_s=1.1, hash_variant=True),
    "fwd_bwd": Workload("fwd_bwd", 8192, 4096, 384, 6, 2048, 2.5, bias_amp=0.01,
                        backward=True),
    "long_slice_fwd_bwd": Workload("long_slice_fwd_bwd", 65536, 4096, 384, 6, 2048, 2.5,
                                   vision_frac=0.30, zipf_s=1.1, backward=True,
                                   recompute=True),
}
ORDER = ["tiny_fwd", "full_fwd", "skewed_mm_fwd", "fwd_bwd", "long_slice_fwd_bwd"]
# the full-width workloads with a shared expert-weight draw (same seed, same shapes)


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(zlib.crc32(f"{seed}:{name}".encode()) & 0x7FFFFFFF)
    return g


def normal_bf16(shape, std, seed, name, device):
    g = _gen(seed, name, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(
        torch.bfloat16)


def stacked_normal_bf16(groups, shape, std, seed, name, device):
    """[groups, *shape] bf16 drawn one group at a time (bounded temporaries)."""
    out = torch.empty((groups, *shape), dtype=torch.bfloat16, device=device)
    g = _gen(seed, name, device)
    for i in range(groups):
        out[i] = (torch.randn(shape, generator=g, device=device, dtype=torch.float32)
                  * std).to(torch.bfloat16)
    return out


def vision_mask(T, frac, seed, device):
    """uint8 [T]: round(frac*T) vision tokens in contiguous blocks of 576 (one
    shorter remainder block), placed at seeded non-overlapping offsets."""
    n_vis = int(round(frac * T))
    mask = torch.zeros(T, dtype=torch.uint8)
    if n_vis == 0:
        return mask.to(device)
    blocks = [VISION_BLOCK] * (n_vis // VISION_BLOCK)
    if n_vis % VISION_BLOCK:
        blocks.append(n_vis % VISION_BLOCK)
    g = _gen(seed, "vision_layout", "cpu")
    order = torch.randperm(len(blocks), generator=g).tolist()
    blocks = [blocks[i] for i in order]
    free = T - n_vis
    # gaps: a uniformly random composition of `free` into len(blocks)+1 parts
    cuts = torch.randperm(free + len(blocks), generator=g)[: len(blocks)].sort().values.tolist()
    pos, prev_cut = 0, -1
    for b, cut in zip(blocks, cuts):
        pos += cut - prev_cut - 1
        mask[pos: pos + b] = 1
        pos += b
        prev_cut = cut
    return mask.to(device)


def zipf_offsets(E, s, seed, device, lam=None):
    """fp32 [E]: offset[e] = -lam * s * ln(rank[e]), rank a seeded permutation of 1..E."""
    lam = ZIPF_LAMBDA if lam is None else lam
    g = _gen(seed, "zipf_rank", "cpu")
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-lam * s * torch.log(rank)).to(torch.float32).to(device)


def zipf_input_ids(T, vocab, s, seed, device):
    """int32 [T]: token ids whose rank frequency follows Zipf(s) over the vocabulary;
    rank -> id through a seeded permutation."""
    g = _gen(seed, "input_ids", "cpu")
    p = torch.arange(1, vocab + 1, dtype=torch.float64).pow(-s)
    ranks = torch.multinomial(p / p.sum(), T, replacement=True, generator=g)
    perm = torch.randperm(vocab, generator=_gen(seed, "vocab_perm", "cpu"))
    return perm[ranks].to(torch.int32).to(device)


def tid2eid_table(vocab, E, k, seed, device):
    """int32 [vocab, k]: k distinct uniformly random experts per token id."""
    g = _gen(seed, "tid2eid", device)
    out = torch.empty((vocab, k), dtype=torch.int32, device=device)
    step = 16384
    for i in range(0, vocab, step):
        n = min(step, vocab - i)
        r = torch.rand((n, E), generator=g, device=device)
        out[i: i + n] = r.topk(k, dim=1).indices.to(torch.int32)
    return out


def make_inputs(w: Workload, device="cpu", with_weights=True, with_dy=None):
    """All inputs of a workload as a dict of tensors on `device`.

    x [T,d] bf16 ~ N(0,1); W_g [E,d], W13 [E+1,2I,d], W2 [E+1,d,I] bf16 ~ N(0,0.02)
    (group E = shared expert); bias [2,E] fp32 ~ U(-bias_amp,bias_amp) (row 0 text, row 1
    vision); is_vision [T] uint8; logit_offset [E] fp32 or None; input_ids [T]
    and tid2eid [VOCAB,k] int32 for the hash variant; dY [T,d] bf16 ~ N(0,1)."""
    s = w.seed
    out = {"x": normal_bf16((w.T, w.d), 1.0, s, "x", device)}
    if with_weights:
        out["W_g"] = normal_bf16((w.E, w.d), 0.02, s, "W_g", device)
        out["W13"] = stacked_normal_bf16(w.E + 1, (2 * w.I, w.d), 0.02, s, "W13", device)
        out["W2"] = stacked_normal_bf16(w.E + 1, (w.d, w.I), 0.02, s, "W2", device)
    gb = _gen(s, "bias", device)
    out["bias"] = ((torch.rand((2, w.E), generator=gb, device=device) * 2.0 - 1.0)
                   * w.bias_amp).float()
    out["is_vision"] = vision_mask(w.T, w.vision_frac, s, device)
    out["logit_offset"] = zipf_offsets(w.E, w.zipf_s, s, device) if w.zipf_s else None
    if w.hash_variant:
        out["input_ids"] = zipf_input_ids(w.T, VOCAB, 1.0, s, device)
        out["tid2eid"] = tid2eid_table(VOCAB, w.E, w.k, s, device)
    if with_dy is None:
        with_dy = w.backward
    if with_dy:
        out["dY"] = normal_bf16((w.T, w.d), 1.0, s, "dY", device)
    return out


def random_ids(T, E, k, seed, device="cpu", skew=0.0):
    """int32 [T,k]: k distinct experts per token (uniform, or skewed towards low
    ids by weights rank^-skew) -- routing decisions as a plain input."""
    g = _gen(seed, "random_ids", "cpu")
    if skew:
        p = torch.arange(1, E + 1, dtype=torch.float64).pow(-skew).expand(T, E)
        ids = torch.multinomial(p, k, replacement=False, generator=g)
    else:
        ids = torch.rand((T, E), generator=g).topk(k, dim=1).indices
    return ids.to(torch.int32).to(device)


def random_logits(T, E, std, seed, device="cpu"):
    """fp32 [T,E] ~ N(0, std^2): gate logits as a plain input."""
    g = _gen(seed, "random_logits", "cpu")
    return (torch.randn((T, E), generator=g, dtype=torch.float32) * std).to(device)
