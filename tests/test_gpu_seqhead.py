"""GPU parity of the DFlash sequential logit head, the confidence head and
confidence pruning (mlx-bun module-dflash.ts: ``#markov`` (Eq 5), ``#rnn``
(Eq 6), ``#confidence`` and the pruning of Alg 1) through fm_draft_pruned,
against the oracle's ``sequential_head`` on the same seeded weights.

Comparison rules: the token of position k must equal the oracle's unless the
oracle's top-2 margin of that position's scores (base logits + bias) is below
1e-3; after an excused difference the later positions follow another prev
token and are not compared.  Confidences agree within 2e-3 (a sigmoid of a
dot product over rows that agree within a relative L2 error of 2e-3).  The
kept length is exact unless the confidence that decides it lies within that
tolerance of its threshold."""
from __future__ import annotations

import math

import numpy as np
import pytest

import fm_synth as S
from gpu_common import MARGIN, REL_L2, Pair, rel_l2
from oracle.common import top2_margin

pytestmark = pytest.mark.gpu

CONF_TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_speculative_decoding_fm_gb300 import build
    build.build()


def small_dflash(**kw):
    c = S.DrafterConfig(S.VARIANT_DFLASH, dim=256, n_heads=2, head_dim=128, n_layers=2, ff_dim=512, block=5,
                        target_dim=320, n_taps=2, vocab=4096, lm_format=S.LM_BF16, max_ctx=160)
    return c.replace(**kw)


def seq_pair(cfg, seed, variant, rank, conf=True):
    def edit(w):
        extra = S.gen_seq_head_weights(cfg, seed, variant, rank=rank)
        if not conf:
            extra = {n: t for n, t in extra.items() if not n.startswith("conf.")}
        w.update(extra)
    return Pair(cfg, seed, keep_hidden=False, edit=edit)


def run_pruned(p, anchor, pos, thresholds=None, min_conf=None, with_conf=True):
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    G = p.cfg.block
    tok = torch.full((G,), -1, dtype=torch.int32, device="cuda")
    conf = torch.full((G,), float("nan"), dtype=torch.float32, device="cuda") if with_conf else None
    length = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    fm.fm_draft_pruned(p.h, 0, anchor, pos, tok, conf, length, thresholds=thresholds, min_conf=min_conf)
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), None if conf is None else conf.cpu().numpy(), int(length.item()))


def thresholds_of(G, thresholds, min_conf):
    mc = math.nan if min_conf is None else float(min_conf)
    if thresholds is None:
        return [mc] * G
    return [float(x) if x is not None and x == x else mc for x in thresholds]


def check_sequential(got_tok, got_conf, got_len, sref, thr):
    """Returns the number of positions compared token for token."""
    n = min(got_len, sref.length)
    assert got_len >= 1 and sref.length >= 1
    for k in range(n):
        if got_conf is not None and len(sref.conf):
            assert abs(float(got_conf[k]) - float(sref.conf[k])) < CONF_TOL, (k, got_conf[k], sref.conf[k])
        if int(got_tok[k]) != int(sref.tokens[k]):
            m = float(top2_margin(sref.scores[k][None])[0])
            assert m < MARGIN, (k, int(got_tok[k]), int(sref.tokens[k]), m)
            return k
    if got_len != sref.length:
        k = n        # the position whose confidence decided differently
        assert k < len(sref.conf) and not math.isnan(thr[k])
        assert abs(float(sref.conf[k]) - thr[k]) < CONF_TOL, (k, got_len, sref.length, sref.conf[k], thr[k])
    return n


@pytest.mark.parametrize("variant", ["markov", "rnn"])
def test_sequential_head_matches_oracle(variant):
    """Several draft cycles without pruning: the tokens through the sequential
    bias, every confidence, length = block; fm_draft on the same handle drafts
    the same tokens; the bias moves some tokens off the parallel argmax."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = small_dflash()
    seed = 1101 if variant == "markov" else 1102
    p = seq_pair(cfg, seed, variant, rank=64)
    fr = S.streams(seed)["features"]
    tr = S.streams(seed)["tokens"]
    p.append(0, S.gen_features(fr, 40, cfg.feat_dim), 0)
    pos, moved, compared = 40, 0, 0
    for cycle in range(6):
        anchor = S.gen_anchor(tr, cfg.vocab)
        tok, conf, length = run_pruned(p, anchor, pos)
        ref = p.oracle.draft(p.state(0), anchor, pos)
        assert rel_l2(p.head_out(), ref.head_out) < REL_L2
        sref = p.oracle.sequential_head(ref, anchor)
        assert sref.length == cfg.block and length == cfg.block
        compared += check_sequential(tok, conf, length, sref, [math.nan] * cfg.block)
        moved += int(np.any(sref.tokens != ref.tokens))
        # fm_draft on a handle with the sequential head drafts through it too
        t2 = torch.zeros((1, cfg.block), dtype=torch.int32, device="cuda")
        fm.fm_draft(p.h, [0], [anchor], [pos], t2)
        torch.cuda.synchronize()
        assert np.array_equal(t2.cpu().numpy()[0], tok)
        n_new = 1 + cycle % 3
        p.append(0, S.gen_features(fr, n_new, cfg.feat_dim), pos)
        pos += n_new
    assert moved >= 1, "the sequential bias never changed a token: the test has no teeth"
    assert compared >= 5 * 6 - 5
    p.close()


@pytest.mark.parametrize("variant", ["markov", "rnn"])
def test_confidence_pruning_matches_oracle(variant):
    """Per-position thresholds and a single min_conf, set from the oracle's
    own confidences so that pruning ends the block at a known position (and at
    none when every threshold is below every confidence)."""
    cfg = small_dflash()
    seed = 1103 if variant == "markov" else 1104
    p = seq_pair(cfg, seed, variant, rank=32)
    fr = S.streams(seed)["features"]
    tr = S.streams(seed)["tokens"]
    p.append(0, S.gen_features(fr, 33, cfg.feat_dim), 0)
    anchor = S.gen_anchor(tr, cfg.vocab)
    ref = p.oracle.draft(p.state(0), anchor, 33)
    base = p.oracle.sequential_head(ref, anchor)
    c = base.conf
    G = cfg.block
    cases = []
    for cut in range(1, G):
        thr = [math.nan] * G
        thr[cut] = float(c[cut]) + 0.05            # prune exactly at cut
        cases.append((thr, None, cut))
    cases.append((None, float(c[1:].min()) - 0.05, G))       # min_conf below every confidence: no pruning
    lo = int(np.argmin(c[1:])) + 1
    first_below = next(k for k in range(1, G) if c[k] < float(c[lo]) + 0.01)
    cases.append((None, float(c[lo]) + 0.01, first_below))   # min_conf just above the lowest confidence
    # position 0 is always kept whatever its threshold
    cases.append(([2.0] + [math.nan] * (G - 1), None, G))
    # a position left open (NaN) takes min_conf: only position 2 can cut
    thr = [0.0] * G
    thr[2] = math.nan
    cases.append((thr, float(c[2]) + 0.05, 2))
    for thresholds, min_conf, want_len in cases:
        sref = p.oracle.sequential_head(ref, anchor, thresholds=thresholds, min_conf=min_conf)
        assert sref.length == want_len
        tok, conf, length = run_pruned(p, anchor, 33, thresholds=thresholds, min_conf=min_conf)
        thr = thresholds_of(G, thresholds, min_conf)
        n = check_sequential(tok, conf, length, sref, thr)
        clear = all(math.isnan(thr[k]) or abs(float(c[k]) - thr[k]) > CONF_TOL for k in range(1, G))
        if n == min(length, want_len) and clear:
            assert length == want_len, (thresholds, min_conf, length, want_len)
        # the cut position's token and confidence are written (its confidence
        # decided the cut); positions after it are not drafted and keep the fill
        assert np.all(tok[length + 1:] == -1) and np.all(np.isnan(conf[length + 1:]))
        assert np.all(tok[:min(length + 1, G)] >= 0) and not np.isnan(conf[:min(length + 1, G)]).any()
    p.close()


def test_sequential_head_errors():
    """fm_draft_pruned needs a sequential head; conf outputs and thresholds
    need a confidence head; nothing is launched when a check fails."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = small_dflash()
    tok = torch.zeros((cfg.block,), dtype=torch.int32, device="cuda")
    conf = torch.zeros((cfg.block,), dtype=torch.float32, device="cuda")
    plain = Pair(cfg, 1105, keep_hidden=False)
    with pytest.raises(fm.FmError) as e:
        fm.fm_draft_pruned(plain.h, 0, 3, 0, tok)
    assert e.value.status == fm.FM_ERR_UNSUPPORTED
    plain.close()
    p = seq_pair(cfg, 1106, "markov", rank=16, conf=False)
    fm.fm_draft_pruned(p.h, 0, 3, 0, tok)                    # no confidence asked: fine
    torch.cuda.synchronize()
    sref = p.oracle.sequential_head(p.oracle.draft(p.state(0), 3, 0), 3)
    check_sequential(tok.cpu().numpy(), None, cfg.block, sref, [math.nan] * cfg.block)
    for kw in ({"conf": conf}, {"min_conf": 0.5}):
        with pytest.raises(fm.FmError) as e:
            fm.fm_draft_pruned(p.h, 0, 3, 0, tok, **kw)
        assert e.value.status == fm.FM_ERR_UNSUPPORTED
    with pytest.raises(fm.FmError) as e:
        fm.fm_draft_pruned(p.h, 0, cfg.vocab, 0, tok)        # anchor outside the vocabulary
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    with pytest.raises(fm.FmError) as e:
        fm.fm_draft_pruned(p.h, 0, 3, 7, tok)                # pos != length
    assert e.value.status == fm.FM_ERR_STATE
    p.close()


def test_sequential_head_full_size():
    """The DFlash-shaped drafter (d 1024, 5 layers, gamma 5, bf16 vocab
    262144) with the Markov head at the pages' rank 256 and the confidence
    head, over a 4096-row context: a few cycles with a min_conf that prunes
    some blocks."""
    cfg = S.dflash_config(max_ctx=4096 + 64)
    seed = 1107
    p = seq_pair(cfg, seed, "markov", rank=256)
    fr = S.streams(seed)["features"]
    tr = S.streams(seed)["tokens"]
    p.append(0, S.gen_features(fr, 4096, cfg.feat_dim), 0)
    pos = 4096
    lengths = []
    for cycle in range(4):
        anchor = S.gen_anchor(tr, cfg.vocab)
        ref = p.oracle.draft(p.state(0), anchor, pos)
        full = p.oracle.sequential_head(ref, anchor)
        min_conf = float(np.median(full.conf[1:]))
        sref = p.oracle.sequential_head(ref, anchor, min_conf=min_conf)
        tok, conf, length = run_pruned(p, anchor, pos, min_conf=min_conf)
        check_sequential(tok, conf, length, sref, [min_conf] * cfg.block)
        lengths.append(length)
        p.append(0, S.gen_features(fr, 2, cfg.feat_dim), pos)
        pos += 2
    assert min(lengths) < cfg.block, lengths
    p.close()
