"""GPU parity of the batched draft: the 16 slot rows of every sequence in a
call go through each product as one tensor-core GEMM (flashmap_drafter.js
``draft`` per anchor; the page hands products above 17 rows to ``runGemm``),
and the cross-attention serves every sequence's own cache in one launch.
Each sequence is checked against the oracle run on its own: the head output
within the relative-L2 bar, the tokens exactly unless the oracle's top-2
margin is below 1e-3, the batched K/V appends through the cache rows, and the
device acceptance bit-exactly."""
from __future__ import annotations

import numpy as np
import pytest

import fm_synth as S
from gpu_common import REL_L2, Pair, rel_l2, tokens_match
from oracle.accept import accept

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_speculative_decoding_fm_gb300 import build
    build.build()


def mid_config(max_seqs: int, max_ctx: int = 400, lm: int = S.LM_Q8_0) -> S.DrafterConfig:
    """FlashMap-shaped, head dim 128 (the batched path's attention), small
    enough for the oracle: D 512, 4 heads, 2 layers, ff 1024, target dim 256,
    2 taps, vocab 4096."""
    return S.DrafterConfig(S.VARIANT_FLASHMAP, dim=512, n_heads=4, head_dim=128, n_layers=2, ff_dim=1024, block=16,
                           target_dim=256, n_taps=2, vocab=4096, lm_format=lm, max_ctx=max_ctx, max_seqs=max_seqs)


def wide_launches(cfg, passes):
    return passes * (3 + 11 * cfg.n_layers + 4)


def head_out(p, seq):
    import block_speculative_decoding_fm_gb300 as fm
    c = p.cfg
    buf = np.empty((c.block, c.target_dim), np.float32)
    fm.fm_debug_copy(p.h, fm.FM_DEBUG_HEAD_OUT, seq, 0, buf)
    return buf


def batched_draft(p, ids, anchors, pos):
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    tok = torch.full((len(ids), p.cfg.block), -1, dtype=torch.int32, device="cuda")
    fm.fm_draft(p.h, ids, anchors, pos, tok)
    torch.cuda.synchronize()
    return tok.cpu().numpy()


def check_seq(p, seq, got_tokens, anchor, pos):
    """One sequence of a batched draft against the oracle's own draft of it:
    head output and logits (the batched lm_head's product, stored instead of
    reduced) within the bar, tokens exact or excused by the margin."""
    import block_speculative_decoding_fm_gb300 as fm
    ref = p.oracle.draft(p.state(seq), anchor, pos)
    y = head_out(p, seq)
    assert rel_l2(y, ref.head_out) < REL_L2, (seq, rel_l2(y, ref.head_out))
    lg = np.empty((p.cfg.block, p.cfg.vocab), np.float32)
    fm.fm_debug_copy(p.h, fm.FM_DEBUG_LOGITS, seq, 0, lg)
    assert rel_l2(lg, ref.logits) < REL_L2, (seq, rel_l2(lg, ref.logits))
    assert tokens_match(got_tokens, ref.tokens, ref.logits), (seq, got_tokens, ref.tokens)
    return ref


def cache_rows_match(p, seq, lo, hi):
    """Cache rows [lo, hi) of every layer against the oracle's f16 rows."""
    st = p.state(seq)
    for l in range(p.cfg.n_layers):
        for which, ref in (("k", st.k[l]), ("v", st.v[l])):
            got = p.cache(seq, l, which)[lo:hi]
            assert rel_l2(got, ref[lo:hi]) < 1e-3, (seq, l, which, rel_l2(got, ref[lo:hi]))


@pytest.mark.parametrize("lm", [S.LM_Q8_0, S.LM_BF16])
def test_batched_cycles_match_oracle(lm):
    """Six sequences with ragged contexts (1 .. 255 rows: several key tiles and
    ragged tails), two draft / accept cycles: a batched append of acc + 1 rows
    per sequence (0 and 16 accepted included), a batched draft, device
    acceptance against seeded targets."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = mid_config(6, lm=lm)
    p = Pair(cfg, 1401, keep_hidden=False)
    fr = S.streams(1401)["features"]
    tr = S.streams(1401)["tokens"]
    lens = [1, 37, 128, 129, 200, 255]
    for s, n in enumerate(lens):
        p.append(s, S.gen_features(fr, n, cfg.feat_dim), 0)
    ids = [3, 0, 5, 1, 4, 2]                   # call order differs from the sequence ids
    length = list(lens)
    acc = [0, 16, 5, 0, 9, 2]                  # accepted last cycle, per call slot
    anchors = [int(tr.integers(0, cfg.vocab)) for _ in ids]
    for cycle in range(2):
        n_new = [a + 1 for a in acc]
        rows = [S.gen_features(fr, n, cfg.feat_dim) for n in n_new]
        fm.fm_context_append_batched(p.h, ids, torch.from_numpy(np.concatenate(rows)).cuda(), n_new,
                                     [length[s] for s in ids])
        for j, s in enumerate(ids):
            p.oracle.context_append(p.state(s), rows[j], length[s])
            length[s] += n_new[j]
        for j, s in enumerate(ids):
            cache_rows_match(p, s, length[s] - n_new[j], length[s])
        pos = [length[s] for s in ids]
        got = batched_draft(p, ids, anchors, pos)
        # one batched pass: prep, anchor_proj, anchor K/V; per layer 11 launches; final adaLN, head,
        # lm_head, row argmax (a per-sequence chain would launch several times as many)
        assert fm.fm_last_launch_count(p.h) == wide_launches(cfg, 1)
        drafts_ok, targets = [], []
        for j, s in enumerate(ids):
            ref = check_seq(p, s, got[j], anchors[j], pos[j])
            drafts_ok.append(bool(np.all(got[j] == ref.tokens)))
            # targets: the oracle's draft with one seeded flip (or none), plus a bonus token
            t = np.append(ref.tokens, int(tr.integers(0, cfg.vocab))).astype(np.int32)
            flip = int(tr.integers(0, cfg.block + 1))
            if flip < cfg.block:
                t[flip] = (t[flip] + 1) % cfg.vocab
            targets.append(t)
        # device acceptance against the oracle's rule
        k = torch.full((len(ids),), cfg.block, dtype=torch.int32, device="cuda")
        a_dev = torch.zeros((len(ids),), dtype=torch.int32, device="cuda")
        b_dev = torch.zeros((len(ids),), dtype=torch.int32, device="cuda")
        fm.fm_accept_batched(p.h, torch.from_numpy(got).cuda(), torch.from_numpy(np.stack(targets)).cuda(), k,
                             a_dev, b_dev)
        torch.cuda.synchronize()
        a_dev, b_dev = a_dev.cpu().numpy(), b_dev.cpu().numpy()
        for j in range(len(ids)):
            if drafts_ok[j]:
                assert (int(a_dev[j]), int(b_dev[j])) == accept(got[j], targets[j], cfg.block)
        acc = [int(a) for a in a_dev]
        anchors = [int(b) for b in b_dev]
    p.close()


def test_batched_draft_in_passes():
    """34 sequences: two batched passes (32 + 2 sequences) in one call, short
    contexts; every sequence's tokens and head output against the oracle."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = mid_config(34, max_ctx=160)
    p = Pair(cfg, 1402, keep_hidden=False)
    fr = S.streams(1402)["features"]
    rng = S.streams(1402)["workload"]
    lens = [int(x) for x in rng.integers(1, 60, size=34)]
    # the contexts through one batched append (no deferred rows are left for the draft to flush)
    rows = [S.gen_features(fr, n, cfg.feat_dim) for n in lens]
    fm.fm_context_append_batched(p.h, list(range(34)), torch.from_numpy(np.concatenate(rows)).cuda(), lens,
                                 [0] * 34)
    for s, n in enumerate(lens):
        p.oracle.context_append(p.state(s), rows[s], 0)
    ids = list(range(34))[::-1]
    anchors = [int(x) for x in rng.integers(0, cfg.vocab, size=34)]
    pos = [lens[s] for s in ids]
    got = batched_draft(p, ids, anchors, pos)
    assert fm.fm_last_launch_count(p.h) == wide_launches(cfg, 2)
    # the first pass's head output has been overwritten by the second pass: reading it is refused
    with pytest.raises(fm.FmError) as e:
        head_out(p, ids[0])
    assert e.value.status == fm.FM_ERR_UNSUPPORTED
    for j, s in enumerate(ids):
        # only the last pass keeps its head output
        if j >= 32:
            check_seq(p, s, got[j], anchors[j], pos[j])
        else:
            ref = p.oracle.draft(p.state(s), anchors[j], pos[j])
            assert tokens_match(got[j], ref.tokens, ref.logits), (s, got[j], ref.tokens)
    p.close()


def test_batched_argmax_ties_go_to_the_lowest_index():
    """Every odd table row copies the even row before it: the lm_head GEMM's
    per-tile best and the row reduction must both keep the even index."""
    def pairs(w):
        t = w["token_embd.weight"]
        t.data = t.data.copy()
        t.data[1::2] = t.data[0::2]
    cfg = mid_config(4, max_ctx=160)
    p = Pair(cfg, 1403, keep_hidden=False, edit=pairs)
    fr = S.streams(1403)["features"]
    lens = [20, 50, 3, 90]
    for s, n in enumerate(lens):
        p.append(s, S.gen_features(fr, n, cfg.feat_dim), 0)
    got = batched_draft(p, [0, 1, 2, 3], [2, 4, 6, 8], lens)
    assert np.all(got % 2 == 0), got
    for s in range(4):
        check_seq(p, s, got[s], [2, 4, 6, 8][s], lens[s])
    p.close()


def test_batched_append_ragged_then_draft():
    """A batched append with ragged row counts: none, one, 127 (the largest that
    takes the shared pass), 33, and 130 (dense: the prefill GEMMs on its own),
    then a batched draft; every sequence against the oracle, the appended cache
    rows included."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = mid_config(5, max_ctx=320)
    p = Pair(cfg, 1405, keep_hidden=False)
    fr = S.streams(1405)["features"]
    base = [20, 3, 90, 1, 40]
    for s, n in enumerate(base):
        p.append(s, S.gen_features(fr, n, cfg.feat_dim), 0)
    add = [0, 1, 127, 33, 130]
    ids = [0, 1, 2, 3, 4]
    rows = [S.gen_features(fr, n, cfg.feat_dim) for n in add]
    fm.fm_context_append_batched(p.h, ids, torch.from_numpy(np.concatenate(rows)).cuda(), add, base)
    for s in ids:
        if add[s]:
            p.oracle.context_append(p.state(s), rows[s], base[s])
        assert fm.fm_get_length(p.h, s) == base[s] + add[s]
        if add[s]:
            cache_rows_match(p, s, base[s], base[s] + add[s])
    pos = [base[s] + add[s] for s in ids]
    anchors = [17, 170, 1700, 4000, 2]
    got = batched_draft(p, ids, anchors, pos)
    assert fm.fm_last_launch_count(p.h) == wide_launches(cfg, 1)
    for s in ids:
        check_seq(p, s, got[s], anchors[s], pos[s])
    p.close()
