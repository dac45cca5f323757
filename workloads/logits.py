"""Seeded synthetic logits and per-row random draws.

Logits for (seed, step, row) come from their own numpy generator, so any subset
of rows of any step can be regenerated on its own (the oracle checks sampled
rows of full-size batches this way).  Values are N(0, sigma); with
``boost_frac > 0`` each token independently (probability ``boost_frac``) gets
``+boost`` before rounding.  ``dtype="bf16"`` rounds the float32 values to
bfloat16 with round-to-nearest-even (torch's conversion) and returns them as
float32 holding exact bf16 values, plus the raw uint16 bit patterns.

``make_logits_device`` draws the same distribution with torch on a device for
the benchmark's resident buffers (a different random stream; only the
distribution matches).
"""

from __future__ import annotations

import numpy as np


def _round_bf16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    vals = t.to(torch.float32).numpy().copy()
    return vals, bits


def make_logits(V: int, rows, step: int, seed: int, sigma: float = 1.0,
                boost: float = 0.0, boost_frac: float = 0.0, dtype: str = "f32"):
    """Return (values f32[len(rows), V], raw) where raw is the device-format array
    (float32 for ``f32``, uint16 bit patterns for ``bf16``)."""
    rows = list(rows)
    out = np.empty((len(rows), V), dtype=np.float32)
    for i, r in enumerate(rows):
        rng = np.random.default_rng([seed, step, r, 0x10617])
        x = rng.normal(0.0, sigma, V).astype(np.float32)
        if boost_frac > 0.0:
            hit = rng.random(V) < boost_frac
            x = np.where(hit, x + np.float32(boost), x).astype(np.float32)
        out[i] = x
    if dtype == "f32":
        return out, out
    if dtype == "bf16":
        return _round_bf16(out)
    raise ValueError(dtype)


def make_logits_device(B: int, V: int, seed: int, sigma: float, boost: float,
                       boost_frac: float, dtype: str, device, generator=None):
    """One [B, V] logits buffer drawn on ``device`` (benchmark inputs)."""
    import torch
    g = generator
    if g is None:
        g = torch.Generator(device=device)
        g.manual_seed(seed)
    x = torch.randn((B, V), generator=g, device=device, dtype=torch.float32) * sigma
    if boost_frac > 0.0:
        hit = torch.rand((B, V), generator=g, device=device) < boost_frac
        x = x + hit.to(torch.float32) * boost
    return x.to(torch.bfloat16) if dtype == "bf16" else x


def make_start_draws(B: int, seed: int) -> np.ndarray:
    """One uniform u32 per row; each side maps it to a start state by its own rule."""
    rng = np.random.default_rng([seed, 0x57A27])
    return rng.integers(0, 2**32, B, dtype=np.uint64).astype(np.uint32)
