"""Pins of the DFlash sequential head and confidence pruning in the oracle
(module-dflash.ts: ``#markov``, ``#rnn``, ``#confidence``, ``forwardRows``)
against a brute-force restatement on micro dims and closed-form special cases.
CPU only."""
from __future__ import annotations

import numpy as np
import pytest

import brute
import fm_synth as S
from oracle import DFlash


def micro(**kw):
    c = S.DrafterConfig(S.VARIANT_DFLASH, dim=8, n_heads=2, head_dim=4, n_layers=2, ff_dim=16, block=3,
                        target_dim=8, n_taps=2, vocab=16, lm_format=S.LM_BF16, max_ctx=24)
    return c.replace(**kw)


def setup(variant, seed, edit=None):
    cfg = micro()
    w = {n: t.data for n, t in S.gen_weights(cfg, seed).items()}
    w.update({n: t.data for n, t in S.gen_seq_head_weights(cfg, seed, variant, rank=4, w1_std=1.0,
                                                            w2_std=0.5).items()})
    if edit:
        edit(w)
    o = DFlash(cfg, w)
    st = o.new_state()
    o.context_append(st, S.gen_features(S.streams(seed)["features"], 5, cfg.feat_dim), 0)
    res = o.draft(st, 3, 5)
    return cfg, w, o, res


@pytest.mark.parametrize("variant", ["markov", "rnn"])
@pytest.mark.parametrize("prune", [None, "thresholds", "min_conf"])
def test_sequential_head_matches_brute_force(variant, prune):
    cfg, w, o, res = setup(variant, 31)
    kw = {}
    if prune == "thresholds":
        kw["thresholds"] = [0.0, 0.5, 0.5]
    elif prune == "min_conf":
        kw["min_conf"] = 0.5
    got = o.sequential_head(res, 3, **kw)
    toks, conf, length = brute.dflash_sequential(w, res.logits.tolist(), res.hidden[-1].tolist(), 3, cfg.rms_eps,
                                                 kw.get("thresholds"), kw.get("min_conf"))
    assert got.length == length
    assert got.tokens.tolist() == toks
    np.testing.assert_allclose(got.conf, conf, rtol=1e-12, atol=1e-14)


def test_sequential_head_changes_some_tokens():
    # the synthetic head is strong enough to move argmaxes (else the parity test would not see it)
    moved = 0
    for seed in range(40, 52):
        cfg, w, o, res = setup("markov", seed)
        moved += int(np.any(o.sequential_head(res, 3).tokens != res.tokens))
    assert moved >= 3


def test_zero_markov_w2_reduces_to_the_parallel_draft():
    def zero(w):
        w["markov.w2"] = np.zeros_like(w["markov.w2"])
    cfg, w, o, res = setup("markov", 32, zero)
    got = o.sequential_head(res, 3)
    assert np.array_equal(got.tokens, res.tokens)
    np.testing.assert_array_equal(got.scores, res.logits)


def test_zero_rnn_output_reduces_to_the_parallel_draft():
    def zero(w):
        w["rnn.wO"] = np.zeros_like(w["rnn.wO"])
    cfg, w, o, res = setup("rnn", 33, zero)
    assert np.array_equal(o.sequential_head(res, 3).tokens, res.tokens)


def test_constant_confidence_and_the_pruning_rule():
    def flat(w):
        w["conf.w"] = np.zeros_like(w["conf.w"])
        w["conf.b"] = S.f32_to_bf16_bits(np.array([0.0], np.float32))    # sigmoid(0) = 1/2
    cfg, w, o, res = setup("markov", 34, flat)
    full = o.sequential_head(res, 3)
    np.testing.assert_array_equal(full.conf, [0.5, 0.5, 0.5])
    assert full.length == 3
    assert o.sequential_head(res, 3, min_conf=0.6).length == 1          # position 0 is always kept
    assert o.sequential_head(res, 3, min_conf=0.4).length == 3
    assert o.sequential_head(res, 3, min_conf=0.5).length == 3          # not below the threshold
    assert o.sequential_head(res, 3, thresholds=[1.0, 0.4, 0.6]).length == 2
    # a given per-position threshold wins over min_conf
    assert o.sequential_head(res, 3, thresholds=[0.0, 0.0, 0.0], min_conf=0.9).length == 3
    # a position the list leaves open (None or NaN) takes min_conf, as the
    # page's per-position lookup falls back to the uniform override
    assert o.sequential_head(res, 3, thresholds=[0.0, None, 0.0], min_conf=0.9).length == 1
    assert o.sequential_head(res, 3, thresholds=[0.0, 0.0, float("nan")], min_conf=0.9).length == 2
    assert o.sequential_head(res, 3, thresholds=[0.0, 0.0], min_conf=0.9).length == 2
    assert o.sequential_head(res, 3, thresholds=[0.0, None, None]).length == 3
