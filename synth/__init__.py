"""Seeded synthetic inputs for the forecast-driven block-sparse decode step.

This module is shared by the tests, the smoke check and the benchmark, for both the CUDA path
and the CPU oracle. It holds none of the method's arithmetic: it draws normal variates,
chooses planted block positions and shifts planted keys along a direction that the caller
supplies. Everything it returns is bfloat16 (torch tensors), the storage type of the decode
step's inputs.

Recipe (per workload, all i.i.d. and seeded):
  * keys, values, queries ~ N(0, 1) bfloat16; hidden states ~ N(0, 1); forecast projection
    weights ~ N(0, 0.02^2); directly drawn forecast vectors ~ N(0, 1);
  * planted blocks: per (layer, sequence, group) ``n_planted`` distinct block indices drawn
    uniformly from 1 .. n_blocks-2 (never block 0 nor the tail block); all 64 keys of each
    planted block are shifted by ``amount * u`` with u the unit vector of the forecast that
    selects that layer's blocks, then rounded back to bfloat16.
"""
from __future__ import annotations

import numpy as np
import torch

BLOCK = 64


def _rng(seed, *stream):
    """A numpy generator for (seed, stream...) so that every tensor has its own stream."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, stream)])))


def normal_bf16(shape, seed, *stream, std=1.0):
    """N(0, std^2) draws, rounded to bfloat16 by torch (round to nearest even), on the CPU."""
    x = _rng(seed, *stream).standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    return torch.from_numpy(x).to(torch.bfloat16)


def normal_bf16_device(shape, seed, device, std=1.0):
    """N(0, std^2) bfloat16 draws made on ``device`` by torch's seeded generator (large
    caches are drawn where they live; tests copy back the slices they check)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # draw in slabs of at most 2^28 elements to bound the float32 temporary
    flat = out.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        n = min(step, flat.numel() - s)
        flat[s:s + n] = (torch.randn(n, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def planted_blocks(seed, n_blocks, n_planted, *stream):
    """``n_planted`` distinct block indices drawn uniformly from 1 .. n_blocks-2, sorted."""
    pool = n_blocks - 2
    if pool <= 0 or n_planted <= 0:
        return np.zeros(0, dtype=np.int64)
    n = min(n_planted, pool)
    return np.sort(_rng(seed, 7, *stream).choice(pool, size=n, replace=False) + 1)


def plant(K, blocks, direction, amount=0.5):
    """Shift every key of the listed blocks by ``amount * direction / |direction|``.

    K: bfloat16 tensor [T, d] (one sequence and group; any device), modified in place.
    blocks: block indices; direction: [d] float tensor or array (any scale; only its
    direction is used).
    """
    if len(blocks) == 0:
        return K
    u = torch.as_tensor(np.asarray(direction, dtype=np.float64))
    u = (u / torch.linalg.vector_norm(u)) * amount
    rows = torch.cat([torch.arange(int(b) * BLOCK, (int(b) + 1) * BLOCK) for b in blocks])
    rows = rows[rows < K.shape[0]].to(K.device)
    K[rows] = (K[rows].double() + u.to(K.device)).to(torch.bfloat16)
    return K


def plant_batched(K, blocks, directions, amount=0.5):
    """Vectorised ``plant`` over a cache K [B, G, T, d] (bfloat16, any device).

    blocks: int array [B, G, n] of planted block indices; directions: float tensor [B, G, d]
    on K's device. One indexed update per call, so that full-size caches plant quickly.
    """
    B, G, T, d = K.shape
    n = blocks.shape[2]
    if n == 0:
        return K
    dev = K.device
    u = directions.to(dev, torch.float64)
    u = u / torch.linalg.vector_norm(u, dim=-1, keepdim=True) * amount          # [B, G, d]
    blk = torch.as_tensor(blocks, device=dev, dtype=torch.int64)                # [B, G, n]
    tok = (blk[..., None] * BLOCK + torch.arange(BLOCK, device=dev)).reshape(B, G, n * BLOCK)
    bg = torch.arange(B * G, device=dev).reshape(B, G, 1).expand(B, G, n * BLOCK)
    flat_rows = (bg * T + tok).reshape(-1)
    shift = u.reshape(B * G, 1, d).expand(B * G, n * BLOCK, d).reshape(-1, d)
    Kf = K.view(B * G * T, d)
    Kf[flat_rows] = (Kf[flat_rows].double() + shift).to(torch.bfloat16)
    return K


def tiny_case(seed, T=4096, B=1, G=2, H=16, d=128, n_planted=8, t_cap=None):
    """The tiny single-layer case: everything ~N(0,1) bf16, forecast drawn directly, planted
    blocks shifted by 0.5 * unit(forecast). K/V hold T tokens (the current one included)."""
    t_cap = t_cap or T
    nb = (T - 1) // BLOCK + 1
    K = normal_bf16((B, G, t_cap, d), seed, 1)
    V = normal_bf16((B, G, t_cap, d), seed, 2)
    q = normal_bf16((B, G * H, d), seed, 3)
    f = normal_bf16((B, G, d), seed, 4)
    planted = np.zeros((B, G, min(n_planted, max(nb - 2, 0))), dtype=np.int64)
    for b in range(B):
        for g in range(G):
            planted[b, g] = planted_blocks(seed, nb, n_planted, b, g)
            plant(K[b, g], planted[b, g], f[b, g].double().numpy())
    return dict(K=K, V=V, q=q, f=f, planted=planted, T=T)


def layer_draws(seed, B, T, G=2, H=16, d=128, hidden=4096, t_cap=None, layer=0):
    """Draws of one 8B-shaped attention layer (before planting): hidden state, forecast
    weights, caches holding T tokens, the decode query and the new token's key/value."""
    t_cap = t_cap or T
    return dict(
        h=normal_bf16((B, hidden), seed, layer, 10),
        W=normal_bf16((G * d, hidden), seed, layer, 11, std=0.02),
        K=normal_bf16((B, G, t_cap, d), seed, layer, 12),
        V=normal_bf16((B, G, t_cap, d), seed, layer, 13),
        q=normal_bf16((B, G * H, d), seed, layer, 14),
        k_new=normal_bf16((B, G, d), seed, layer, 15),
        v_new=normal_bf16((B, G, d), seed, layer, 16),
    )
