"""FlashMap drafter forward pass, plain fp64 (oracle).  TEST INFRASTRUCTURE:
see oracle/common.py for who may use this package.

Source: diskformer 0.5.4 -> 0.6.6, package/engines/flashmap_drafter.js -- the
header comment (the math of the drafter), ``init`` (h0), ``extendContext``
(context injection) and ``draft`` (the 16-slot block, head, lm_head, argmax).
The tied token table E [V, Ht] is the target's table (bf16 or Q8_0).

Readings taken where the page leaves a step open:
  * anchor_proj, x_embed, mlp.fc1/fc2 and head carry biases; fc, every q/k/v/o
    projection and the context k/v projections have none (the page's ``gemm``
    adds a bias only when the checkpoint has one, and passes ``false`` for the
    bias-free ones).
  * modulation block n (n = 3l + {0 self, 1 cross, 2 mlp}, n = 3L final) is
    [scale D | shift D | gate D].
  * context row r sits at position r, the anchor at ``pos``, block slot t at
    ``pos + 1 + t``; cross-attention reads cache rows 0..pos (the anchor's own
    slot included).
  * the cache stores f16 (``kvWrite``); every other activation is exact.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Mapping

import numpy as np

from .common import (attention, bf16_to_f64, f16_store, gelu_erf, head_rms_norm, layer_norm_modulate,
                     linear, q8_0_dequant, rms_norm, rope_interleaved)


@dataclass
class FlashMapState:
    """One sequence's context: per layer the f16-valued key and value rows
    (position-major, [max_ctx, D]) and the number of valid rows."""
    k: List[np.ndarray]
    v: List[np.ndarray]
    length: int = 0


@dataclass
class DraftResult:
    tokens: np.ndarray                 # [B] int64
    logits: np.ndarray                 # [B, V]
    head_out: np.ndarray               # Y [B, Ht]
    hidden: List[np.ndarray] = field(default_factory=list)   # X after each layer [B, D]


class FlashMap:
    def __init__(self, cfg, weights: Mapping[str, np.ndarray], modulation: np.ndarray, table_q8: bool):
        """cfg: any object with the DrafterConfig fields (dim, n_heads, ...).
        weights: name -> raw storage (bf16 bit patterns as uint16; the token
        table as uint16 bf16 bits or uint8 Q8_0 blocks when ``table_q8``).
        modulation: [(3L + 1) * 3 * D] f32."""
        self.cfg = cfg
        D = cfg.dim
        self.w: Dict[str, np.ndarray] = {}
        for name, arr in weights.items():
            if name == "token_embd.weight":
                continue
            self.w[name] = bf16_to_f64(arr)
        raw = weights["token_embd.weight"]
        self.E = q8_0_dequant(raw, cfg.target_dim) if table_q8 else bf16_to_f64(raw)
        self.mod = np.asarray(modulation, dtype=np.float64).reshape(3 * cfg.n_layers + 1, 3, D)
        self.h0 = self._initial_state()

    # -- init: the constant input of every slot at zero noise ---------------
    def _initial_state(self) -> np.ndarray:
        """h0 = x_embed(state_norm(uniform_embeds)), uniform_embeds = the mean
        row of E (flashmap_drafter.js header, ``init``: colMeanQ8 -> rmsRows ->
        x_embed)."""
        c = self.cfg
        u = self.E.mean(axis=0)[None, :]
        s = rms_norm(u, self.w["state_norm.weight"], c.rms_eps)
        return linear(s, self.w["x_embed.weight"], self.w["x_embed.bias"])[0]

    def new_state(self, max_ctx: int | None = None) -> FlashMapState:
        c = self.cfg
        n = max_ctx or c.max_ctx
        # f16 values are exact in f32, so the cache is held as f32
        return FlashMapState([np.zeros((n, c.dim), np.float32) for _ in range(c.n_layers)],
                             [np.zeros((n, c.dim), np.float32) for _ in range(c.n_layers)], 0)

    def _kv_rows(self, l: int, x: np.ndarray, positions: np.ndarray):
        """Cross-attention key/value rows of layer l for normalised context
        rows x: k = RoPE(k_norm(k_proj x)), v = v_proj x (no bias)."""
        c = self.cfg
        p = f"layers.{l}.cross_attn."
        k = linear(x, self.w[p + "k_proj.weight"])
        v = linear(x, self.w[p + "v_proj.weight"])
        k = head_rms_norm(k, self.w[p + "k_norm.weight"], c.qk_eps, c.head_dim)
        k = rope_interleaved(k, positions, c.head_dim, c.rope_theta)
        return k, v

    # -- extendContext ------------------------------------------------------
    def context_append(self, st: FlashMapState, feats: np.ndarray, start: int) -> None:
        """Append feature rows [n, taps * Ht] as positions start .. start+n-1:
        fc -> hidden_norm -> per layer k/v (``extendContext``)."""
        c = self.cfg
        n = feats.shape[0]
        if start < 0 or start > st.length:
            raise ValueError("start beyond the context")
        if start + n + c.block + 1 > st.k[0].shape[0]:
            raise ValueError("context full")
        x = linear(np.asarray(feats, np.float64), self.w["fc.weight"])
        x = rms_norm(x, self.w["hidden_norm.weight"], c.rms_eps)
        pos = start + np.arange(n)
        for l in range(c.n_layers):
            k, v = self._kv_rows(l, x, pos)
            st.k[l][start:start + n] = f16_store(k)
            st.v[l][start:start + n] = f16_store(v)
        st.length = start + n

    # -- draft --------------------------------------------------------------
    def draft(self, st: FlashMapState, anchor: int, pos: int) -> DraftResult:
        """The ``block`` tokens after ``anchor`` at context position ``pos``
        (``draft``): anchor slot -> block of h0 -> L DiT layers -> final adaLN
        -> head -> lm_head (E^T) -> argmax."""
        c = self.cfg
        D, B, hd = c.dim, c.block, c.head_dim
        if pos != st.length:
            raise ValueError("pos must equal the context length")
        if pos + c.block + 1 > st.k[0].shape[0]:
            raise ValueError("context full")
        # the anchor's context slot
        e = self.E[anchor][None, :]
        a = linear(e, self.w["anchor_proj.weight"], self.w["anchor_proj.bias"])
        a = rms_norm(a, self.w["anchor_norm.weight"], c.rms_eps)
        for l in range(c.n_layers):
            k, v = self._kv_rows(l, a, np.array([pos]))
            st.k[l][pos] = f16_store(k)[0]
            st.v[l][pos] = f16_store(v)[0]
        L = pos + 1
        # the jump 0 -> 1 from zero noise: every slot starts at h0
        X = np.tile(self.h0[None, :], (B, 1))
        spos = pos + 1 + np.arange(B)
        hidden = []
        for l in range(c.n_layers):
            p = f"layers.{l}."
            # self-attention over the block (no mask)
            m = self.mod[3 * l + 0]
            H = layer_norm_modulate(X, m[0], m[1], c.ln_eps)
            q = linear(H, self.w[p + "self_attn.q_proj.weight"])
            k = linear(H, self.w[p + "self_attn.k_proj.weight"])
            v = linear(H, self.w[p + "self_attn.v_proj.weight"])
            q = rope_interleaved(head_rms_norm(q, self.w[p + "self_attn.q_norm.weight"], c.qk_eps, hd),
                                 spos, hd, c.rope_theta)
            k = rope_interleaved(head_rms_norm(k, self.w[p + "self_attn.k_norm.weight"], c.qk_eps, hd),
                                 spos, hd, c.rope_theta)
            o = attention(q, k, v, hd)
            X = X + m[2] * linear(o, self.w[p + "self_attn.o_proj.weight"])
            # cross-attention over the cached context rows 0..pos
            m = self.mod[3 * l + 1]
            H = layer_norm_modulate(X, m[0], m[1], c.ln_eps)
            q = linear(H, self.w[p + "cross_attn.q_proj.weight"])
            q = rope_interleaved(head_rms_norm(q, self.w[p + "cross_attn.q_norm.weight"], c.qk_eps, hd),
                                 spos, hd, c.rope_theta)
            o = attention(q, st.k[l][:L].astype(np.float64), st.v[l][:L].astype(np.float64), hd)
            X = X + m[2] * linear(o, self.w[p + "cross_attn.o_proj.weight"])
            # MLP: fc1 -> exact GELU -> fc2
            m = self.mod[3 * l + 2]
            H = layer_norm_modulate(X, m[0], m[1], c.ln_eps)
            u = gelu_erf(linear(H, self.w[p + "mlp.fc1.weight"], self.w[p + "mlp.fc1.bias"]))
            X = X + m[2] * linear(u, self.w[p + "mlp.fc2.weight"], self.w[p + "mlp.fc2.bias"])
            hidden.append(X.copy())
        m = self.mod[3 * c.n_layers]
        H = layer_norm_modulate(X, m[0], m[1], c.ln_eps)
        Y = linear(H, self.w["head.weight"], self.w["head.bias"])
        logits = Y @ self.E.T
        tokens = np.argmax(logits, axis=-1).astype(np.int64)
        return DraftResult(tokens, logits, Y, hidden)
