"""The MTP (multi-token prediction) draft head, plain fp64 (oracle).
TEST INFRASTRUCTURE: see oracle/common.py for who may use this package.

Source: diskformer 0.5.3 -> 0.6.4, package/engines/ternary_bonsai_2_mtp.js --
the header's graph description, ``MCFG``, the kernels ``WG_NORM``,
``WG_QKPREP``, ``WG_ATTN``, ``WG_SILU_MUL``, ``WG_Q8`` and ``MTPHead.forward``,
and ``MTPRunner``'s draft loop (the first pass over the pending rows, then one
single-row pass per further depth step).

One forward over M rows (tokens x at positions pos0 .. pos0 + M - 1, each with
h, the normed hidden of the previous position):
  Xc = [rms(E[x]; enorm) | rms(h; hnorm)];  X = eh_proj Xc
  A = rms(X; attn_norm);  Qf = attn_q A  (per q head 2 * hd: the query, then a gate)
  K = attn_k A, V = attn_v A  (n_kv heads)
  per head: RMSNorm over hd (attn_q_norm / attn_k_norm), then NEOX RoPE on the
  first rot dims (pairs i, i + rot/2, angle pos * theta^(-2i / rot)); the K and
  V rows go to the head's own cache at their positions
  O[m, h] = softmax_j(q . k_j / sqrt(hd)) v_j over cache rows kv_lo .. pos0 + m
  (kv head h // (n_heads / n_kv)), times sigmoid(gate[m, h])
  X += attn_output O;  A = rms(X; post_attention_norm)
  X += ffn_down(silu(ffn_gate A) * ffn_up A);  h' = rms(X; shared_head_norm)
  draft = argmax(lm_head h')
Depth chaining: the next pass takes the draft token and h' of the last row.

Readings taken where the page leaves a step open:
  * the embedding table and the lm_head are the trunk's; here they are a plain
    bf16 embedding table and a Q8_0 lm_head (the trunk stores its lm_head
    ternary behind a Hadamard rotation, a storage format the head's math does
    not see).
  * the RoPE angle is exact (the page forms it in f32).
  * the K/V cache is exact (the page keeps it f32).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Mapping

import numpy as np

from .common import bf16_to_f64, q8_0_dequant, rms_norm

Q8_MATRICES = ("eh_proj", "attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up", "ffn_down")
NORMS = ("enorm", "hnorm", "attn_norm", "attn_q_norm", "attn_k_norm", "post_attention_norm", "shared_head_norm")


@dataclass
class MtpState:
    k: np.ndarray      # [cap, n_kv * hd]
    v: np.ndarray


@dataclass
class MtpPass:
    hout: np.ndarray   # [M, H] shared_head_norm output
    x_attn: np.ndarray  # [M, H] X after the attention residual
    gated: np.ndarray  # [M, n_heads * hd] the gated attention output


def neox_rope(x: np.ndarray, pos: int, rot: int, theta: float) -> np.ndarray:
    """Rotate pairs (i, i + rot/2), i < rot/2, of one head vector by
    pos * theta^(-2i / rot); dims from rot on are left as they are
    (``WG_QKPREP``: NEOX RoPE on the first 64 of 256 dims)."""
    out = np.array(x, dtype=np.float64)
    half = rot // 2
    i = np.arange(half, dtype=np.float64)
    a = float(pos) * theta ** (-2.0 * i / rot)
    c, s = np.cos(a), np.sin(a)
    x0, x1 = out[:half].copy(), out[half:rot].copy()
    out[:half] = x0 * c - x1 * s
    out[half:rot] = x1 * c + x0 * s
    return out


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x), as ``WG_SILU_MUL`` writes it: g / (1 + exp(-g))."""
    return x / (1.0 + np.exp(-x))


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


class MtpHead:
    def __init__(self, cfg, weights: Mapping[str, np.ndarray]):
        """weights: the Q8_0 matrices as raw GGUF rows ([N][K/32 * 34] uint8,
        y = W x with W [N][K]), the norms as f32, ``token_embd`` as bf16 bits
        [V][H] and ``lm_head`` as Q8_0 rows [V][H / 32 * 34]."""
        self.cfg = cfg
        c = cfg
        ks = {"eh_proj": 2 * c.hidden, "attn_q": c.hidden, "attn_k": c.hidden, "attn_v": c.hidden,
              "attn_output": c.n_heads * c.head_dim, "ffn_gate": c.hidden, "ffn_up": c.hidden, "ffn_down": c.inter}
        self.w = {n: q8_0_dequant(weights[n], ks[n]) for n in Q8_MATRICES}
        for n in NORMS:
            self.w[n] = np.asarray(weights[n], dtype=np.float64)
        self.embd = weights["token_embd"]          # bf16 bits, rows decoded on use
        self.lm_raw = weights["lm_head"]           # Q8_0 rows, dequantised by row blocks on use

    def new_state(self, cap: int | None = None) -> MtpState:
        c = self.cfg
        n = cap or c.kv_cap
        return MtpState(np.zeros((n, c.n_kv_heads * c.head_dim)), np.zeros((n, c.n_kv_heads * c.head_dim)))

    def embed(self, tokens) -> np.ndarray:
        return bf16_to_f64(self.embd[np.asarray(tokens, dtype=np.int64)])

    def forward(self, st: MtpState, embed: np.ndarray, hn: np.ndarray, pos0: int, kv_lo: int) -> MtpPass:
        """``MTPHead.forward`` over M = len(embed) rows at positions pos0..;
        writes their K/V cache rows."""
        c, w = self.cfg, self.w
        M = embed.shape[0]
        hd, nh, nkv = c.head_dim, c.n_heads, c.n_kv_heads
        xc = np.concatenate([rms_norm(embed, w["enorm"], c.eps), rms_norm(hn, w["hnorm"], c.eps)], axis=1)
        x = xc @ w["eh_proj"].T
        a = rms_norm(x, w["attn_norm"], c.eps)
        qf = a @ w["attn_q"].T
        kt = a @ w["attn_k"].T
        vt = a @ w["attn_v"].T
        q = np.zeros((M, nh, hd))
        for m in range(M):
            pos = pos0 + m
            for h in range(nh):
                qh = rms_norm(qf[m, h * 2 * hd:h * 2 * hd + hd], w["attn_q_norm"], c.eps)
                q[m, h] = neox_rope(qh, pos, c.rot_dims, c.theta)
            for g in range(nkv):
                kh = rms_norm(kt[m, g * hd:(g + 1) * hd], w["attn_k_norm"], c.eps)
                st.k[pos, g * hd:(g + 1) * hd] = neox_rope(kh, pos, c.rot_dims, c.theta)
            st.v[pos] = vt[m]
        gated = np.zeros((M, nh * hd))
        group = nh // nkv
        for m in range(M):
            last = pos0 + m
            for h in range(nh):
                g = h // group
                keys = st.k[kv_lo:last + 1, g * hd:(g + 1) * hd]
                vals = st.v[kv_lo:last + 1, g * hd:(g + 1) * hd]
                s = keys @ q[m, h] / np.sqrt(hd)
                p = np.exp(s - s.max())
                o = (p / p.sum()) @ vals
                gate = qf[m, h * 2 * hd + hd:(h + 1) * 2 * hd]
                gated[m, h * hd:(h + 1) * hd] = o * sigmoid(gate)
        x = x + gated @ w["attn_output"].T
        x_attn = x.copy()
        a = rms_norm(x, w["post_attention_norm"], c.eps)
        f = silu(a @ w["ffn_gate"].T) * (a @ w["ffn_up"].T)
        x = x + f @ w["ffn_down"].T
        return MtpPass(rms_norm(x, w["shared_head_norm"], c.eps), x_attn, gated)

    def logits(self, hout: np.ndarray, rows_per_block: int = 8192) -> np.ndarray:
        """lm_head over the whole vocabulary, dequantised a block of rows at a time."""
        c = self.cfg
        out = np.empty((hout.shape[0], c.vocab))
        for r0 in range(0, c.vocab, rows_per_block):
            blk = q8_0_dequant(self.lm_raw[r0:r0 + rows_per_block], c.hidden)
            out[:, r0:r0 + blk.shape[0]] = hout @ blk.T
        return out

    def draft(self, st: MtpState, tokens, hn: np.ndarray, pos0: int, kv_lo: int, depth: int):
        """``MTPRunner``'s draft: a pass over the M pending rows (tokens at
        pos0.., hn their previous-position hiddens), the argmax of the last
        row's head output, then depth - 1 single-row passes, each on the
        previous draft token and the previous pass's last h'.
        Returns (drafts [depth], logits of each drafted position [depth][V],
        the h' rows of each pass)."""
        tokens = list(tokens)
        res = self.forward(st, self.embed(tokens), np.asarray(hn, dtype=np.float64), pos0, kv_lo)
        lg = [self.logits(res.hout[-1:])[0]]
        drafts = [int(np.argmax(lg[0]))]
        houts: List[np.ndarray] = [res.hout]
        pos = pos0 + len(tokens)
        for d in range(1, depth):
            res = self.forward(st, self.embed([drafts[-1]]), houts[-1][-1:], pos, kv_lo)
            lg.append(self.logits(res.hout)[0])
            drafts.append(int(np.argmax(lg[-1])))
            houts.append(res.hout)
            pos += 1
        return np.array(drafts, np.int64), np.stack(lg), houts
