"""Parity at the full workload sizes, in the launch configuration bench.py
times: the FlashMap-Qwen3-4B-shaped step (1024 cached rows, append 17, draft
at 1041) and DFlash-shaped draft/accept cycles over a 4096-row context."""
from __future__ import annotations

import numpy as np
import pytest

import fm_synth as S
from gpu_common import REL_L2, Pair, rel_l2, tokens_match

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_speculative_decoding_fm_gb300 import build
    build.build()


def test_flashmap_4b_step():
    cfg = S.flashmap_4b_config()
    p = Pair(cfg, 1002)
    fr = S.streams(1002)["features"]
    p.append(0, S.gen_features(fr, 1024, cfg.feat_dim), 0)
    f17 = S.gen_features(fr, 17, cfg.feat_dim)
    p.append(0, f17, 1024)
    anchor = S.gen_anchor(S.streams(1002)["tokens"], cfg.vocab)
    got, ref = p.draft(0, anchor, 1041)
    for l in range(cfg.n_layers):
        assert rel_l2(p.hidden(l), ref.hidden[l]) < REL_L2, l
    assert rel_l2(p.head_out(), ref.head_out) < REL_L2
    lg = p.logits()
    assert rel_l2(lg, ref.logits) < REL_L2
    assert tokens_match(got, ref.tokens, ref.logits), (got, ref.tokens)
    st = p.state(0)
    for l in (0, cfg.n_layers - 1):
        for which, want in (("k", st.k[l]), ("v", st.v[l])):
            c = p.cache(0, l, which)
            rows = [0, 1, 511, 1023, 1024, 1040, 1041]
            assert rel_l2(c[rows], want[rows]) < 1e-3
    # a second step from the same state (rewind to 1024) is bit-identical
    p.append(0, f17, 1024, oracle=False)
    got2, _ = p.draft(0, anchor, 1041, oracle=False)
    assert np.array_equal(got, got2)
    p.close()


def test_dflash_cycles_full_size():
    cfg = S.dflash_config()
    p = Pair(cfg, 1004)
    fr = S.streams(1004)["features"]
    tr = S.streams(1004)["tokens"]
    p.append(0, S.gen_features(fr, 4096, cfg.feat_dim), 0)
    pos, anchor = 4096, S.gen_anchor(tr, cfg.vocab)
    from oracle import accept
    for cycle in range(4):
        got, ref = p.draft(0, anchor, pos)
        if cycle == 0:
            for l in range(cfg.n_layers):
                assert rel_l2(p.hidden(l), ref.hidden[l]) < REL_L2, l
            assert rel_l2(p.logits(), ref.logits) < REL_L2
        assert rel_l2(p.head_out(), ref.head_out) < REL_L2
        assert tokens_match(got, ref.tokens, ref.logits), (cycle, got, ref.tokens)
        acc = int(tr.integers(0, cfg.block + 1))
        target = S.targets_with_flip(ref.tokens, cfg.block, acc, cfg.vocab, tr)
        n_acc, bonus = accept(ref.tokens, target, cfg.block)
        assert n_acc == acc
        p.append(0, S.gen_features(fr, n_acc + 1, cfg.feat_dim), pos)
        pos += n_acc + 1
        anchor = bonus
    p.close()


def test_long_context_prefill_and_draft():
    """32768 context rows through the dense prefill, then one draft over 32769 keys."""
    cfg = S.flashmap_4b_config(max_ctx=32768 + 64)
    p = Pair(cfg, 1003)
    fr = S.streams(1003)["features"]
    feats = S.gen_features(fr, 32768, cfg.feat_dim)
    p.append(0, feats, 0)
    st = p.state(0)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(32768, 64, replace=False))
    for l in range(cfg.n_layers):
        for which, want in (("k", st.k[l]), ("v", st.v[l])):
            got = p.cache(0, l, which)
            assert rel_l2(got[rows], want[rows]) < 1e-3, (l, which)
    anchor = S.gen_anchor(S.streams(1003)["tokens"], cfg.vocab)
    got, ref = p.draft(0, anchor, 32768)
    assert rel_l2(p.head_out(), ref.head_out) < REL_L2
    assert tokens_match(got, ref.tokens, ref.logits), (got, ref.tokens)
    p.close()
