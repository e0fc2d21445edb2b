"""Time conditioning of the FlashMap drafter, plain fp64 (oracle).
TEST INFRASTRUCTURE: see oracle/common.py for who may use this package.

Source: diskformer 0.5.4 -> 0.6.6, package/engines/flashmap_drafter.js --
``timeConditioning`` (the adaLN table of the jump s -> t, computed once at
``init`` with s = 0, t = 1) and ``CFG`` (timeDim, timeScale, cond).

For a time value x the page forms a sinusoidal embedding of width timeDim:
with half = timeDim / 2 and frequencies f_i = exp(-ln(10000) i / half),
e[i] = cos(x * timeScale * f_i) and e[half + i] = sin(x * timeScale * f_i).
That embedding goes through two linears with a SiLU between them
(``time_embed`` for s, ``jump_embed`` for t); cond = SiLU(ts + tj).  Each
adaLN linear maps cond to one [scale D | shift D | gate D] block, in the order
(self, cross, mlp) of every layer, then the final norm.

Readings taken where the page leaves a step open:
  * SiLU(x) = x / (1 + exp(-x)), as the page writes it.
  * the page rounds the frequency and the angle to f32 (JS typed arrays); the
    oracle keeps them exact, as it does for the RoPE angles.
  * linears carry a bias when the checkpoint has one; a missing bias is zero.
"""
from __future__ import annotations

from typing import Mapping

import numpy as np

from .common import bf16_to_f64, linear


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x), written as the page does: x / (1 + exp(-x))."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def sinusoidal_embedding(time: float, time_dim: int, time_scale: float) -> np.ndarray:
    """[cos(a_0) .. cos(a_{half-1}) | sin(a_0) .. sin(a_{half-1})] with
    a_i = time * time_scale * exp(-ln(10000) i / half) (``timeConditioning``'s
    ``embed``)."""
    half = time_dim // 2
    i = np.arange(half, dtype=np.float64)
    f = np.exp(-np.log(10000.0) * i / half)
    a = (time * time_scale) * f
    return np.concatenate([np.cos(a), np.sin(a)])


def adaln_names(n_layers: int):
    """The adaLN linears in table order: (self, cross, mlp) per layer, then the final norm."""
    names = []
    for l in range(n_layers):
        for n in ("self_attn_adaln", "cross_attn_adaln", "mlp_adaln"):
            names.append(f"layers.{l}.{n}.linear")
    names.append("final_adaln.linear")
    return names


def time_conditioning(weights: Mapping[str, np.ndarray], n_layers: int, dim: int, time_dim: int,
                      time_scale: float, s: float, t: float) -> np.ndarray:
    """The adaLN table [(3 n_layers + 1) * 3 * dim] of the jump s -> t.
    weights: name -> bf16 bit patterns (uint16) of ``time_embed.linear_{1,2}``,
    ``jump_embed.linear_{1,2}`` and every adaLN linear (``.weight`` [out][in],
    optional ``.bias``)."""
    w = {n: bf16_to_f64(a) for n, a in weights.items()}

    def lin(name, x):
        return linear(x[None, :], w[name + ".weight"], w.get(name + ".bias"))[0]

    def embed(prefix, time):
        e = sinusoidal_embedding(time, time_dim, time_scale)
        return lin(prefix + ".linear_2", silu(lin(prefix + ".linear_1", e)))

    cond = silu(embed("time_embed", s) + embed("jump_embed", t))
    out = [lin(name, cond) for name in adaln_names(n_layers)]
    table = np.concatenate(out)
    assert table.shape == ((3 * n_layers + 1) * 3 * dim,)
    return table
