"""Plain fp64 building blocks of the drafter oracle.

TEST INFRASTRUCTURE.  This package is the slow, obviously-correct CPU
restatement of what the drafter computes, used only to check the CUDA path.
Only tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline leg
(and its ``--impl reference`` arm) may import it.  It shares no code with the
CUDA library and the library never calls it.

Sources (page title, file, section):
  [FM]  diskformer 0.5.4 -> 0.6.6, package/engines/flashmap_drafter.js
  [MTP] diskformer 0.5.3 -> 0.6.4, package/engines/ternary_bonsai_2_mtp.js
  [DF]  mlx-bun 0.4.0 -> 1.0.0, package/src/spec/dspark/module-dflash.ts

Every function below is a definition written out in float64 with numpy; a
matrix product or a reduction is a library call, nothing is blocked or fused.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf as _erf


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> value: the f32 whose high half is the pattern
    ([FM] WGSL helper ``bf``: f32 = bits << 16)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f16_store(x: np.ndarray) -> np.ndarray:
    """The context cache holds f16 ([FM] ``kvWrite``: cache = f16(k), f16(v));
    the value read back is x rounded to the nearest f16."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def q8_0_dequant(raw: np.ndarray, ncols: int) -> np.ndarray:
    """Rows of GGUF Q8_0 blocks -> values.  Each 34-byte block is a
    little-endian f16 scale d followed by 32 int8 q; value = d * q
    ([MTP] ``loadWeights``, ggml type 8; [FM] ``colMeanQ8`` reads the same
    scale-times-int8 product)."""
    raw = np.asarray(raw, dtype=np.uint8)
    rows = raw.shape[0]
    nb = ncols // 32
    blk = raw.reshape(rows, nb, 34)
    d = np.ascontiguousarray(blk[:, :, 0:2]).view("<f2").astype(np.float64)   # [rows, nb, 1]
    q = np.ascontiguousarray(blk[:, :, 2:34]).view(np.int8).astype(np.float64)  # [rows, nb, 32]
    return (d * q).reshape(rows, ncols)


def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """y[t, m] = sum_k x[t, k] w[m, k] (+ b[m]); w is [out][in]
    ([FM] ``gemmBf16``: y[t*M + m] = sum_k x[t*N + k] W[m][k] + b[m])."""
    y = x @ w.T
    return y + b if b is not None else y


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y = x * w / sqrt(mean(x^2) + eps) over the last axis
    ([FM] ``rmsRows``; [DF] ``ops.rmsNorm`` with a plain weight)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def layer_norm_modulate(x: np.ndarray, scale: np.ndarray, shift: np.ndarray, eps: float) -> np.ndarray:
    """adaLN: LayerNorm without affine (population variance, divide by D),
    then * (1 + scale) + shift ([FM] ``lnMod``)."""
    mu = np.mean(x, axis=-1, keepdims=True)
    var = np.mean((x - mu) ** 2, axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * (1.0 + scale) + shift


def head_rms_norm(x: np.ndarray, w: np.ndarray, eps: float, head_dim: int) -> np.ndarray:
    """Per-head RMSNorm over head_dim with a head_dim-long weight indexed by
    channel ([FM] ``headNormRope``, first half).  x: [T, n_heads * head_dim]."""
    T = x.shape[0]
    xh = x.reshape(T, -1, head_dim)
    return rms_norm(xh, w, eps).reshape(T, -1)


def rope_angles(positions: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """a[t, i] = p_t * theta^(-2i / head_dim), i < head_dim / 2, in float64
    ([FM] ``ropeRows``; the page rounds the angle to f32, the oracle keeps it
    exact)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / head_dim)
    return np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]


def rope_interleaved(x: np.ndarray, positions: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """Rotate interleaved channel pairs (2i, 2i+1) of every head by the angle
    of the row's position ([FM] ``headNormRope``, second half):
    (x0, x1) -> (x0 cos a - x1 sin a, x1 cos a + x0 sin a)."""
    T = x.shape[0]
    xh = x.reshape(T, -1, head_dim)
    a = rope_angles(positions, head_dim, theta)[:, None, :]   # [T, 1, hd/2]
    c, s = np.cos(a), np.sin(a)
    x0 = xh[:, :, 0::2]
    x1 = xh[:, :, 1::2]
    out = np.empty_like(xh)
    out[:, :, 0::2] = x0 * c - x1 * s
    out[:, :, 1::2] = x1 * c + x0 * s
    return out.reshape(T, -1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, head_dim: int) -> np.ndarray:
    """Unmasked multi-head attention: per head softmax(q k^T / sqrt(hd)) v.
    q [Tq, h*hd], k, v [Tk, h*hd] -> [Tq, h*hd]  ([FM] ``attn``; [DF] ``sdpa``
    with scale hd^-1/2 and no mask)."""
    Tq, Tk = q.shape[0], k.shape[0]
    qh = q.reshape(Tq, -1, head_dim)
    kh = k.reshape(Tk, -1, head_dim)
    vh = v.reshape(Tk, -1, head_dim)
    s = np.einsum("qhd,khd->hqk", qh, kh) / np.sqrt(head_dim)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    o = np.einsum("hqk,khd->qhd", p, vh)
    return o.reshape(Tq, -1)


def gelu_erf(x: np.ndarray) -> np.ndarray:
    """Exact GELU x * Phi(x) = x/2 (1 + erf(x / sqrt 2)) ([FM] ``gelu``; the
    page evaluates erf with a 1.5e-7 approximation, the oracle exactly)."""
    return 0.5 * x * (1.0 + _erf(x / np.sqrt(2.0)))


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """tanh-approximate GELU ([DF] ``ops.geluApprox`` in the gated FFN):
    x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """Per-row argmax; ties go to the lowest index (first occurrence)."""
    return np.argmax(logits, axis=-1).astype(np.int64)


def top2_margin(logits: np.ndarray) -> np.ndarray:
    """Per-row gap between the largest and second-largest logit."""
    part = np.partition(logits, -2, axis=-1)
    return part[..., -1] - part[..., -2]
