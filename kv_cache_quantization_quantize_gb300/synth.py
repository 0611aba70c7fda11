"""Seeded synthetic K/V/Q workloads. Only random numbers and shapes live here; the quantization
method does not.

The shapes stand in for Llama-3.1-8B (32 layers, 32 query heads, 8 KV heads, head_dim 128, GQA 4:1)
and for a head_dim-256 model. No weights or datasets are involved.

Draw order for one (layer) call, from one torch.Generator seeded with ``seed``:
1. K ~ dist.
2. V ~ dist.
3. The outlier channels of K, per KV head: ``randperm(d)[:m]``, scaled by ``factor``.
4. Q ~ N(0, 1).

Distributions:
* ``normal`` is N(0, 1).
* ``student_t5`` is a Student-t with nu=5, divided by sqrt(5/3) to give unit variance.
"""

import torch

__all__ = ["kv_tokens", "queries", "ragged_lengths"]


def _draw(gen, shape, dist, device):
    if dist == "normal":
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if dist == "student_t5":
        nu = 5.0
        z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        # chi-square(5) as a sum of 5 squared normals keeps the draw inside one generator
        chi = torch.zeros(shape, device=device, dtype=torch.float32)
        for _ in range(5):
            chi += torch.randn(shape, generator=gen, device=device, dtype=torch.float32) ** 2
        return z / torch.sqrt(chi / nu) / (nu / (nu - 2.0)) ** 0.5
    raise ValueError(dist)


def kv_tokens(n_tokens, n_heads, d, *, seed, dist="normal", outliers=None, dtype=torch.bfloat16,
              device="cpu", gen=None):
    """K, V of shape [n_tokens, n_heads, d].

    ``outliers`` is None, ("fixed", channels, factor) or ("random", m, factor): K channels scaled per head.
    """
    if gen is None:
        gen = torch.Generator(device=device)
        gen.manual_seed(int(seed))
    shape = (n_tokens, n_heads, d)
    k = _draw(gen, shape, dist, device)
    v = _draw(gen, shape, dist, device)
    if outliers is not None:
        kind, what, factor = outliers
        for h in range(n_heads):
            if kind == "fixed":
                ch = torch.tensor(list(what), device=device)
            else:
                ch = torch.randperm(d, generator=gen, device=device)[:int(what)]
            k[:, h, ch] *= float(factor)
    return k.to(dtype), v.to(dtype)


def queries(batch, n_q_heads, d, *, seed, dtype=torch.bfloat16, device="cpu", gen=None):
    """Q ~ N(0, 1) of shape [batch, n_q_heads, d]."""
    if gen is None:
        gen = torch.Generator(device=device)
        gen.manual_seed(int(seed) + 7919)
    return torch.randn((batch, n_q_heads, d), generator=gen, device=device, dtype=torch.float32).to(dtype)


def ragged_lengths(batch, lo, hi, *, seed):
    """Integer lengths uniform in [lo, hi] inclusive (CPU generator)."""
    gen = torch.Generator()
    gen.manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (batch,), generator=gen).tolist()
