"""Shared set-up of the GPU parity tests: build a drafter through the C ABI
and the oracle on the same seeded inputs, and the comparison rules."""
from __future__ import annotations

import numpy as np

import block_speculative_decoding_fm_gb300 as fm
import fm_synth as S
from oracle import DFlash, FlashMap
from oracle.common import top2_margin

# Parity bars (the drafter's stated tolerance): hidden states and logits within
# a relative L2 error of 2e-3; draft tokens exact except where the oracle's
# top-2 logit margin is below 1e-3; acceptance bit-exact.
REL_L2 = 2e-3
MARGIN = 1e-3


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def tokens_match(got, want, logits) -> bool:
    got = np.asarray(got)
    want = np.asarray(want)
    margin = top2_margin(np.asarray(logits))
    return bool(np.all((got == want) | (margin < MARGIN)))


def persistent_step_requested() -> bool:
    """FM_PERSISTENT=1 asks fm_create for the one-launch draft step."""
    import os
    return os.environ.get("FM_PERSISTENT", "") == "1"


class Pair:
    """The CUDA drafter (through the C ABI) and the oracle on one workload."""

    def __init__(self, cfg: S.DrafterConfig, seed: int, oracle_max_ctx: int | None = None, keep_hidden=True,
                 edit=None):
        """edit: optional callable that changes the generated weights (name ->
        fm_synth.Tensor) in place before both sides are built."""
        import torch
        self.torch = torch
        self.cfg = cfg
        self.seed = seed
        self.w = S.gen_weights(cfg, seed)
        if edit is not None:
            edit(self.w)
        raw = {n: t.data for n, t in self.w.items()}
        if cfg.variant == S.VARIANT_FLASHMAP:
            self.mod = S.gen_modulation(cfg, seed)
            self.oracle = FlashMap(cfg, raw, self.mod, cfg.lm_format == S.LM_Q8_0)
        else:
            self.mod = None
            self.oracle = DFlash(cfg, raw)
        self.h = fm.fm_create(cfg, fm.weight_items(self.w), self.mod)
        if keep_hidden:
            fm.fm_set_debug(self.h, fm.FM_DEBUG_KEEP_HIDDEN)
        self.states = {}
        self.oracle_max_ctx = oracle_max_ctx or cfg.max_ctx

    def state(self, seq):
        if seq not in self.states:
            self.states[seq] = self.oracle.new_state(self.oracle_max_ctx)
        return self.states[seq]

    def append(self, seq, feats: np.ndarray, start: int, oracle=True):
        t = self.torch.from_numpy(np.ascontiguousarray(feats, np.float32)).cuda()
        fm.fm_context_append(self.h, seq, t, feats.shape[0], start)
        if oracle:
            self.oracle.context_append(self.state(seq), feats, start)

    def draft(self, seq, anchor, pos, oracle=True):
        tok = self.torch.zeros((1, self.cfg.block), dtype=self.torch.int32, device="cuda")
        fm.fm_draft(self.h, [seq], [anchor], [pos], tok)
        self.last_launches = fm.fm_last_launch_count(self.h)
        self.torch.cuda.synchronize()
        got = tok.cpu().numpy()[0]
        ref = self.oracle.draft(self.state(seq), anchor, pos) if oracle else None
        return got, ref

    def hidden(self, layer):
        out = np.empty((self.cfg.block, self.cfg.dim), np.float32)
        return fm.fm_debug_copy(self.h, fm.FM_DEBUG_HIDDEN, 0, layer, out)

    def head_out(self, seq=0):
        out = np.empty((self.cfg.block, self.cfg.target_dim), np.float32)
        return fm.fm_debug_copy(self.h, fm.FM_DEBUG_HEAD_OUT, seq, 0, out)

    def logits(self, seq=0):
        out = np.empty((self.cfg.block, self.cfg.vocab), np.float32)
        return fm.fm_debug_copy(self.h, fm.FM_DEBUG_LOGITS, seq, 0, out)

    def cache(self, seq, layer, which="k"):
        c = self.cfg
        out = np.empty((c.n_heads, c.max_ctx, c.head_dim), np.float16)
        fm.fm_debug_copy(self.h, fm.FM_DEBUG_CACHE_K if which == "k" else fm.FM_DEBUG_CACHE_V, seq, layer, out)
        return out.transpose(1, 0, 2).reshape(c.max_ctx, c.dim).astype(np.float32)

    def close(self):
        fm.fm_destroy(self.h)
        self.h = None
