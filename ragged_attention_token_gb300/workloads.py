"""Seeded synthetic inputs for the pack -> attend -> unpack path.

This module only draws random numbers: keep masks and Q/K/V values with the
shapes, dtypes and length mixes of DeiT attention layers after token pruning.
It holds none of the method's arithmetic (no packing, no attention) and it is
the single piece of code shared by the CPU oracle's tests and the CUDA path's
tests and benchmark, so both sides always see identical input bits.

Workloads (DeiT attention shapes, head_dim 64, CLS token at position 0):

  tiny         B=2,   N=197, H=3,  fp16; per-image keep rate r_b ~ U[0.2,1.0],
               every patch kept ~ Bernoulli(r_b), CLS always kept.
  serving      B in {1,2,4}, N=197, H=6, bf16; 80% pruning: n_b ~ UniformInt[35,43]
               tokens incl. CLS, the n_b-1 patches drawn without replacement.
  batched      B=64,  N=197, H=12, bf16; pruning p in {0,.5,.8,.9}:
               n_b = 1 + clamp(round(196*(1-p)*(1+u_b)), 0, 196), u_b ~ U[-.1,.1]
               (p = 0 keeps all 197 tokens, no jitter).
  hires        B=32,  N=577, H=12, bf16; p in {.5,.8,.9}, same rule over 576 patches.
  progressive  B=256, N=197, H=6,  bf16, 12 layers; before layers 4, 7 and 10 each
               image keeps CLS plus the top ceil(0.7*m) of its m surviving patches by
               a U[0,1) score (ties to the lower index); pruned tokens stay pruned,
               so every image has 197/139/98/69 tokens; fresh Q/K/V every layer.

Values are N(0,1) drawn in fp32 by a seeded torch CPU generator and rounded to
the input dtype (round-to-nearest-even).  Seeds are ``1000*workload + sub``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 64

WORKLOADS = ("tiny", "serving", "batched", "hires", "progressive")
_WORKLOAD_INDEX = {name: i + 1 for i, name in enumerate(WORKLOADS)}
_CHAIN_SEED_BASE = 1_000_000   # seeds of the progressive chain: base + 100*B (+ layer)

SERVING_BATCHES = (1, 2, 4)
BATCHED_RATES = (0.0, 0.5, 0.8, 0.9)
HIRES_RATES = (0.5, 0.8, 0.9)
PROGRESSIVE_LAYERS = 12
PROGRESSIVE_EVENTS = (4, 7, 10)   # 1-indexed layers whose input is pruned
PROGRESSIVE_KEEP = 0.7


@dataclass
class Case:
    """One batch of synthetic input for one attention layer."""
    name: str
    B: int
    N: int
    H: int
    d: int
    dtype: torch.dtype
    keep: torch.Tensor            # uint8 [B, N], nonzero = keep
    q: torch.Tensor               # [B, N, H, d] in ``dtype``
    k: torch.Tensor
    v: torch.Tensor
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def lengths(self) -> list[int]:
        return [int(x) for x in (self.keep != 0).sum(dim=1).tolist()]

    @property
    def kept_tokens(self) -> int:
        return int((self.keep != 0).sum().item())


def seed_for(workload: str, sub: int = 0) -> int:
    return 1000 * _WORKLOAD_INDEX[workload] + sub


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _values(g: torch.Generator, B: int, N: int, H: int, d: int, dtype: torch.dtype):
    out = []
    for _ in range(3):
        x = torch.randn((B, N, H, d), generator=g, dtype=torch.float32)
        out.append(x.to(dtype).contiguous())
    return out


def _mask_from_counts(g: torch.Generator, counts: list[int], N: int) -> torch.Tensor:
    """CLS (position 0) kept; ``counts[b] - 1`` patches drawn without replacement."""
    B = len(counts)
    keep = torch.zeros((B, N), dtype=torch.uint8)
    for b, n in enumerate(counts):
        if n <= 0:
            continue
        keep[b, 0] = 1
        if n > 1:
            perm = torch.randperm(N - 1, generator=g)[: n - 1] + 1
            keep[b, perm] = 1
    return keep


def jittered_counts(g: torch.Generator, B: int, patches: int, rate: float) -> list[int]:
    """n_b = 1 + clamp(round(patches*(1-rate)*(1+u_b)), 0, patches), u_b ~ U[-0.1, 0.1].

    A rate of 0 keeps every token (no jitter): the dense case.
    """
    if rate == 0.0:
        return [patches + 1] * B
    u = torch.rand((B,), generator=g, dtype=torch.float64) * 0.2 - 0.1
    out = []
    for b in range(B):
        m = int(round(patches * (1.0 - rate) * (1.0 + float(u[b]))))
        out.append(1 + min(max(m, 0), patches))
    return out


def make_tiny(seed: int | None = None) -> Case:
    seed = seed_for("tiny") if seed is None else seed
    g = _gen(seed)
    B, N, H = 2, 197, 3
    r = torch.rand((B,), generator=g, dtype=torch.float64) * 0.8 + 0.2
    u = torch.rand((B, N), generator=g, dtype=torch.float64)
    keep = (u < r[:, None]).to(torch.uint8)
    keep[:, 0] = 1
    q, k, v = _values(g, B, N, H, HEAD_DIM, torch.float16)
    return Case("tiny", B, N, H, HEAD_DIM, torch.float16, keep, q, k, v, seed,
                {"keep_rate": r.tolist()})


def make_serving(B: int = 4, seed: int | None = None) -> Case:
    if B not in SERVING_BATCHES and seed is None:
        raise ValueError(f"serving batch must be one of {SERVING_BATCHES}")
    seed = seed_for("serving", SERVING_BATCHES.index(B) if B in SERVING_BATCHES else 9) if seed is None else seed
    g = _gen(seed)
    N, H = 197, 6
    counts = torch.randint(35, 44, (B,), generator=g).tolist()
    keep = _mask_from_counts(g, counts, N)
    q, k, v = _values(g, B, N, H, HEAD_DIM, torch.bfloat16)
    return Case(f"serving_B{B}", B, N, H, HEAD_DIM, torch.bfloat16, keep, q, k, v, seed,
                {"pruning": 0.8})


def make_batched(rate: float = 0.8, seed: int | None = None) -> Case:
    sub = BATCHED_RATES.index(rate) if rate in BATCHED_RATES else 9
    seed = seed_for("batched", sub) if seed is None else seed
    g = _gen(seed)
    B, N, H = 64, 197, 12
    counts = jittered_counts(g, B, N - 1, rate)
    keep = _mask_from_counts(g, counts, N)
    q, k, v = _values(g, B, N, H, HEAD_DIM, torch.bfloat16)
    return Case(f"batched_p{int(rate * 100)}", B, N, H, HEAD_DIM, torch.bfloat16, keep, q, k, v,
                seed, {"pruning": rate})


def make_hires(rate: float = 0.8, seed: int | None = None) -> Case:
    sub = HIRES_RATES.index(rate) if rate in HIRES_RATES else 9
    seed = seed_for("hires", sub) if seed is None else seed
    g = _gen(seed)
    B, N, H = 32, 577, 12
    counts = jittered_counts(g, B, N - 1, rate)
    keep = _mask_from_counts(g, counts, N)
    q, k, v = _values(g, B, N, H, HEAD_DIM, torch.bfloat16)
    return Case(f"hires_p{int(rate * 100)}", B, N, H, HEAD_DIM, torch.bfloat16, keep, q, k, v,
                seed, {"pruning": rate})


def progressive_masks(B: int = 256, N: int = 197, seed: int | None = None) -> list[torch.Tensor]:
    """Keep mask of each of the 12 layers of the progressive-pruning workload.

    Scores are drawn once per (event, image, token).  At an event every image
    keeps CLS and the top ceil(0.7*m) of its m surviving patches; sorting is
    stable on the descending score so equal scores keep the lower index.
    """
    seed = seed_for("progressive") if seed is None else seed
    g = _gen(seed)
    scores = torch.rand((len(PROGRESSIVE_EVENTS), B, N), generator=g, dtype=torch.float32)
    keep = torch.ones((B, N), dtype=torch.uint8)
    masks = []
    event = 0
    for layer in range(1, PROGRESSIVE_LAYERS + 1):
        if layer in PROGRESSIVE_EVENTS:
            new = torch.zeros_like(keep)
            new[:, 0] = keep[:, 0]
            for b in range(B):
                alive = torch.nonzero(keep[b, 1:], as_tuple=False).flatten() + 1
                m = int(alive.numel())
                k_top = int(math.ceil(PROGRESSIVE_KEEP * m))
                s = scores[event, b, alive]
                order = torch.sort(s, descending=True, stable=True).indices
                new[b, alive[order[:k_top]]] = 1
            keep = new
            event += 1
        masks.append(keep.clone())
    return masks


def make_progressive_layer(layer: int, masks: list[torch.Tensor] | None = None,
                           seed: int | None = None) -> Case:
    """Layer ``layer`` (1-indexed) of the progressive workload: its mask and fresh Q/K/V."""
    if not 1 <= layer <= PROGRESSIVE_LAYERS:
        raise ValueError("layer is 1-indexed, 1..12")
    B, N, H = 256, 197, 6
    masks = progressive_masks(B, N) if masks is None else masks
    seed = seed_for("progressive", layer) if seed is None else seed
    g = _gen(seed)
    q, k, v = _values(g, B, N, H, HEAD_DIM, torch.bfloat16)
    return Case(f"progressive_L{layer}", B, N, H, HEAD_DIM, torch.bfloat16,
                masks[layer - 1].clone(), q, k, v, seed, {"layer": layer})


def make_progressive_chain(B: int = 256, N: int = 197, H: int = 6,
                           seed: int | None = None) -> tuple[list[torch.Tensor], list[Case]]:
    """The 12-layer progressive workload at batch B as one chain: the masks of
    ``progressive_masks(B, N)`` and, per layer, fresh seeded Q/K/V.  The chained
    path packs layer 1 from its padded tensors and re-packs every later layer's
    inputs from the previous layer's packed layout."""
    base = _CHAIN_SEED_BASE + 100 * B if seed is None else seed
    masks = progressive_masks(B, N, base)
    cases = []
    for layer in range(1, PROGRESSIVE_LAYERS + 1):
        g = _gen(base + layer)
        q, k, v = _values(g, B, N, H, HEAD_DIM, torch.bfloat16)
        cases.append(Case(f"progressive_chain_L{layer}", B, N, H, HEAD_DIM, torch.bfloat16,
                          masks[layer - 1].clone(), q, k, v, base + layer, {"layer": layer}))
    return masks, cases


def make_custom(B: int, N: int, H: int, lengths: list[int] | None = None,
                dtype: torch.dtype = torch.bfloat16, seed: int = 12345,
                random_mask: bool = False, value_scale: float = 1.0,
                cls: bool = True) -> Case:
    """Edge-case generator: explicit per-image kept counts, or a Bernoulli(1/2) mask.

    With ``cls`` the first kept token is position 0 (for counts >= 1).
    """
    g = _gen(seed)
    if random_mask:
        keep = (torch.rand((B, N), generator=g) < 0.5).to(torch.uint8)
    else:
        assert lengths is not None and len(lengths) == B
        if cls:
            keep = _mask_from_counts(g, list(lengths), N)
        else:
            keep = torch.zeros((B, N), dtype=torch.uint8)
            for b, n in enumerate(lengths):
                if n > 0:
                    keep[b, torch.randperm(N, generator=g)[:n]] = 1
    q, k, v = _values(g, B, N, H, HEAD_DIM, dtype)
    if value_scale != 1.0:
        q = (q.float() * value_scale).to(dtype)
    return Case(f"custom_B{B}_N{N}_H{H}", B, N, H, HEAD_DIM, dtype, keep, q, k, v, seed,
                {"value_scale": value_scale})


def all_cases(include_progressive: bool = True) -> list[Case]:
    """Every (workload, sub-case) pair at full size."""
    cases = [make_tiny()]
    cases += [make_serving(B) for B in SERVING_BATCHES]
    cases += [make_batched(p) for p in BATCHED_RATES]
    cases += [make_hires(p) for p in HIRES_RATES]
    if include_progressive:
        masks = progressive_masks()
        cases += [make_progressive_layer(L, masks) for L in range(1, PROGRESSIVE_LAYERS + 1)]
    return cases
