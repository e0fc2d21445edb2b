"""DFlash / DSpark KV-injection drafter forward pass, plain fp64 (oracle).
TEST INFRASTRUCTURE: see oracle/common.py for who may use this package.

Source: mlx-bun 0.4.0 -> 1.0.0, package/src/spec/dspark/module-dflash.ts --
header (Eq 2, Eq 3), ``#buildContext`` (Eq 2), ``projectContextRows`` (the
retained per-layer context K/V), ``#buildBlock``, ``#layer`` (Eq 3),
``#backbone``, ``#baseLogits`` and the greedy branch of ``forwardRows``.
Weights are [in, out] as the page stores them (y = x @ W).

Readings taken where the page leaves a step open:
  * eps is the target's RMSNorm eps; the page takes it from the target config;
    1e-6 here.
  * the anchor embedding is a plain row of the tied token table E (no scale);
    the bf16 cast of the hidden before the target's lm_head is not modelled.
  * the retained context K/V is kept exact (the page keeps it as an f32 array).
  * ``draft`` is the parallel draft, the base logits' argmax (what the page
    drafts while markov.w2 is still at its zero init); ``sequential_head``
    adds the sequential bias, the confidence and the pruning on top of it.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Mapping

import numpy as np

from .common import attention, bf16_to_f64, gelu_tanh, rms_norm


@dataclass
class SequentialResult:
    tokens: np.ndarray            # [gamma] greedy tokens with the sequential bias
    scores: np.ndarray            # [gamma, V] base logits + bias
    conf: np.ndarray              # [gamma] predicted acceptance (empty without a confidence head)
    length: int                   # positions kept after confidence pruning (gamma without pruning)


@dataclass
class DFlashState:
    k: List[np.ndarray]      # per layer [max_ctx, d]
    v: List[np.ndarray]
    length: int = 0


@dataclass
class DFlashResult:
    tokens: np.ndarray            # [gamma]
    logits: np.ndarray            # [gamma, V]
    head_out: np.ndarray          # out_proj output [gamma, H]
    hidden: List[np.ndarray] = field(default_factory=list)   # H_d after each layer


class DFlash:
    def __init__(self, cfg, weights: Mapping[str, np.ndarray]):
        self.cfg = cfg
        self.w: Dict[str, np.ndarray] = {n: bf16_to_f64(a) for n, a in weights.items()}
        self.E = self.w.pop("token_embd.weight")

    def new_state(self, max_ctx: int | None = None) -> DFlashState:
        c = self.cfg
        n = max_ctx or c.max_ctx
        return DFlashState([np.zeros((n, c.dim)) for _ in range(c.n_layers)],
                           [np.zeros((n, c.dim)) for _ in range(c.n_layers)], 0)

    def build_context(self, feats: np.ndarray) -> np.ndarray:
        """Eq 2: H_ctx = RMSNorm(F W_c; ctx_norm)."""
        c = self.cfg
        return rms_norm(np.asarray(feats, np.float64) @ self.w["W_c"], self.w["ctx_norm"], c.rms_eps)

    def context_append(self, st: DFlashState, feats: np.ndarray, start: int) -> None:
        """Retain per layer K_i = attn_norm_i(H_ctx) W_k,i and V likewise
        (``projectContextRows``) for rows start .. start+n-1."""
        c = self.cfg
        n = feats.shape[0]
        if start < 0 or start > st.length:
            raise ValueError("start beyond the context")
        if start + n + c.block + 1 > st.k[0].shape[0]:
            raise ValueError("context full")
        h = self.build_context(feats)
        for i in range(c.n_layers):
            nc = rms_norm(h, self.w[f"bb.{i}.attn_norm"], c.rms_eps)
            st.k[i][start:start + n] = nc @ self.w[f"bb.{i}.k"]
            st.v[i][start:start + n] = nc @ self.w[f"bb.{i}.v"]
        st.length = start + n

    def build_block(self, anchor: int) -> np.ndarray:
        """Row 0 = tok_proj(E[anchor]) + block_pos[0]; row j = mask_emb[j-1] +
        block_pos[j] (``#buildBlock``)."""
        c = self.cfg
        bp = self.w["block_pos"]
        rows = [self.E[anchor] @ self.w["tok_proj"] + bp[0]]
        for j in range(1, c.block):
            rows.append(self.w["mask_emb"][j - 1] + bp[j])
        return np.stack(rows)

    def layer(self, i: int, Hd: np.ndarray, Kc: np.ndarray, Vc: np.ndarray) -> np.ndarray:
        """Eq 3 (``#layer``): the block attends bidirectionally over
        [context ++ block] with the layer's own W_k / W_v on both; no mask, no
        RoPE; plain residuals; gated GELU(tanh) FFN."""
        c = self.cfg
        w = self.w
        p = f"bb.{i}."
        nd = rms_norm(Hd, w[p + "attn_norm"], c.rms_eps)
        q = nd @ w[p + "q"]
        kd = nd @ w[p + "k"]
        vd = nd @ w[p + "v"]
        o = attention(q, np.concatenate([Kc, kd]), np.concatenate([Vc, vd]), c.head_dim)
        H = Hd + o @ w[p + "o"]
        n2 = rms_norm(H, w[p + "ff_norm"], c.rms_eps)
        return H + (gelu_tanh(n2 @ w[p + "gate"]) * (n2 @ w[p + "up"])) @ w[p + "down"]

    def draft(self, st: DFlashState, anchor: int, pos: int) -> DFlashResult:
        """gamma tokens after ``anchor`` given the retained context rows
        0..pos-1 (``#backbone`` -> ``#baseLogits`` -> argmax per position)."""
        c = self.cfg
        if pos != st.length:
            raise ValueError("pos must equal the context length")
        L = pos
        Hd = self.build_block(anchor)
        hidden = []
        for i in range(c.n_layers):
            Hd = self.layer(i, Hd, st.k[i][:L], st.v[i][:L])
            hidden.append(Hd.copy())
        out = rms_norm(Hd, self.w["out_norm"], c.rms_eps)
        Y = out @ self.w["out_proj"]
        logits = Y @ self.E.T
        return DFlashResult(np.argmax(logits, axis=-1).astype(np.int64), logits, Y, hidden)

    def sequential_head(self, res: DFlashResult, anchor: int, thresholds=None, min_conf=None) -> SequentialResult:
        """The sequential logit head and confidence pruning of the greedy draft
        (``forwardRows``: ``#markov`` / ``#rnn`` per position, ``#confidence``,
        Alg 1 pruning).  For position k, with prev the anchor (k = 0) or the token
        of position k - 1:
          e1 = markov.w1[prev];
          Markov: bias = e1 markov.w2;  RNN: s = tanh(s rnn.wH + e1 + rnn.bH)
          (s starts at 0), bias = s rnn.wO;
          token_k = argmax(base logits_k + bias);
          conf_k = sigmoid([block_k, e1] conf.w + conf.b), block = the
          out_norm'd backbone rows.
        Pruning: the threshold of position k is thresholds[k] when the list has
        one there (not None, not NaN), else min_conf (the page's
        ``thresholds?.[step] ?? minConf``); the block ends at the first k >= 1
        whose conf_k is below it (position 0 is always kept), and no later
        position is drafted."""
        c = self.cfg
        w = self.w
        rnn = "rnn.wH" in w
        has_conf = "conf.w" in w
        block = rms_norm(res.hidden[-1], w["out_norm"], c.rms_eps)
        r = w["markov.w1"].shape[1]
        state = np.zeros(r)
        prev = int(anchor)
        tokens, scores, conf = [], [], []
        length = None
        for k in range(c.block):
            e1 = w["markov.w1"][prev]
            if rnn:
                state = np.tanh(state @ w["rnn.wH"] + e1 + w["rnn.bH"])
                bias = state @ w["rnn.wO"]
            else:
                bias = e1 @ w["markov.w2"]
            sc = res.logits[k] + bias
            tok = int(np.argmax(sc))
            tokens.append(tok)
            scores.append(sc)
            prev = tok
            if has_conf:
                z = float(np.concatenate([block[k], e1]) @ w["conf.w"][:, 0] + w["conf.b"][0])
                conf.append(1.0 / (1.0 + np.exp(-z)))
                thr = thresholds[k] if thresholds is not None and k < len(thresholds) else None
                if thr is None or thr != thr:      # no threshold of its own (None or NaN): min_conf
                    thr = min_conf
                if k > 0 and thr is not None and conf[-1] < thr:
                    length = k
                    break
        if length is None:
            length = len(tokens)
        return SequentialResult(np.array(tokens, np.int64), np.stack(scores), np.array(conf), length)
