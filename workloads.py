"""Seeded synthetic inputs for the embedding weight-gradient workloads.

Shared by the tests, the smoke check and the bench, for both the CUDA path and the
oracle.  It holds none of the method's arithmetic: it only draws token ids and
normally distributed gradient / main_grad values.

Recipe (the same for every workload):
  * seed = 1000 + the workload's index in WORKLOADS;
  * ids are drawn with numpy's PCG64 from that seed.  "uniform" draws integers in
    [0, V).  "zipf" draws ranks k = 1..V with P(k) proportional to k**-s by inverse CDF
    in float64 (searchsorted of uniform draws into the normalised cumulative pmf), and
    uses id = k - 1, so the hot ids are the small ones;
  * "forced" (long runs): a fraction of the positions, chosen without replacement,
    is set to the last id V - 1, which is cold under the Zipf draw, so it forms one long
    run of its own;
  * grad ~ N(0, grad_std) and main_grad ~ N(0, mg_std) (the number is the standard
    deviation), drawn in float32 by a torch.Generator seeded from the same seed on
    the device the tensor is made on, then cast to the workload's dtype.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_embeddings: int          # V
    hidden: int                  # H
    ids_shape: tuple             # grad is [*ids_shape, H]
    ids_dist: str                # "uniform" | "zipf"
    zipf_s: float = 0.0
    forced_fraction: float = 0.0
    grad_dtype: torch.dtype = torch.bfloat16
    grad_std: float = 1.0
    mg_dtype: torch.dtype = torch.float32
    mg_std: float = 1.0
    index: int = 0

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def num_tokens(self) -> int:
        return int(np.prod(self.ids_shape))


WORKLOADS = [
    Workload("tiny", 1024, 256, (4096,), "uniform", grad_std=1.0, mg_std=0.01, index=0),
    Workload("gpt2_like", 50257, 1024, (4, 2048), "zipf", zipf_s=1.1, grad_std=1e-2,
             mg_std=1e-3, index=1),
    Workload("large_vocab", 129280, 7168, (1, 8192), "zipf", zipf_s=1.1, grad_std=1e-2,
             mg_std=1e-3, index=2),
    Workload("long_runs", 129280, 7168, (65536,), "zipf", zipf_s=1.3, forced_fraction=0.2,
             grad_std=1e-2, mg_dtype=torch.bfloat16, mg_std=1e-3, index=3),
    Workload("big_batch", 256000, 8192, (16, 8192), "uniform", grad_std=1e-2, mg_std=1e-3,
             index=4),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def zipf_ids(rng: np.random.Generator, V: int, s: float, size: int) -> np.ndarray:
    """Bounded Zipf(s) over ids 0..V-1 (id = rank - 1), inverse CDF in float64."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    pmf = ranks ** (-s)
    cdf = np.cumsum(pmf)
    cdf /= cdf[-1]
    u = rng.random(size)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int64)


def make_ids(w: Workload) -> np.ndarray:
    """int64 ids with shape w.ids_shape."""
    rng = np.random.default_rng(w.seed)
    n = w.num_tokens
    if w.ids_dist == "uniform":
        ids = rng.integers(0, w.num_embeddings, size=n, dtype=np.int64)
    elif w.ids_dist == "zipf":
        ids = zipf_ids(rng, w.num_embeddings, w.zipf_s, n)
    else:
        raise ValueError(w.ids_dist)
    if w.forced_fraction > 0:
        k = int(round(w.forced_fraction * n))
        where = rng.choice(n, size=k, replace=False)
        ids[where] = w.num_embeddings - 1
    return ids.reshape(w.ids_shape)


def normal(shape, std: float, dtype: torch.dtype, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std) in float32 from a seeded generator on `device`, cast to `dtype`."""
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    x.mul_(std)
    return x.to(dtype)


def make_grad(w: Workload, device="cpu") -> torch.Tensor:
    return normal((*w.ids_shape, w.hidden), w.grad_std, w.grad_dtype, w.seed * 7 + 1, device)


def make_main_grad(w: Workload, device="cpu") -> torch.Tensor:
    return normal((w.num_embeddings, w.hidden), w.mg_std, w.mg_dtype, w.seed * 7 + 2, device)


def scaled(w: Workload, num_embeddings=None, hidden=None, num_tokens=None) -> Workload:
    """The same recipe at other sizes (tests use it to shrink a workload)."""
    shape = w.ids_shape if num_tokens is None else (num_tokens,)
    return dataclasses.replace(w, num_embeddings=num_embeddings or w.num_embeddings,
                               hidden=hidden or w.hidden, ids_shape=shape)
