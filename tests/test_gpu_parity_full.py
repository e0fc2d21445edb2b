"""Parity at the full workload sizes, in the launch configuration bench.py
times: the FlashMap-Qwen3-4B-shaped step (1024 cached rows, append 17, draft
at 1041) and DFlash-shaped draft/accept cycles over a 4096-row context."""
from __future__ import annotations

import numpy as np
import pytest

import fm_synth as S
from gpu_common import REL_L2, Pair, persistent_step_requested, rel_l2, tokens_match

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
    if persistent_step_requested():
        assert p.last_launches <= 6, p.last_launches      # anchor, K/V, the step, the lm_head
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
    """The DFlash-shaped workload over its 200 draft / accept cycles: every
    cycle's tokens and head output against the oracle, the logits every 40th
    cycle, and the acceptance of every cycle computed on the device by
    fm_accept_batched (bit-exact with the acceptance rule on the same drafts
    and with the seeded acceptance count when the drafts equal the oracle's).
    Both sides then append acc + 1 fresh rows at the anchor position."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    from oracle import accept
    cfg = S.dflash_config()
    p = Pair(cfg, 1004)
    fr = S.streams(1004)["features"]
    tr = S.streams(1004)["tokens"]
    p.append(0, S.gen_features(fr, 4096, cfg.feat_dim), 0)
    pos, anchor = 4096, S.gen_anchor(tr, cfg.vocab)
    G = cfg.block
    k_dev = torch.full((1,), G, dtype=torch.int32, device="cuda")
    acc_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    bonus_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    same = 0
    for cycle in range(200):
        got, ref = p.draft(0, anchor, pos)
        if cycle == 0:
            for l in range(cfg.n_layers):
                assert rel_l2(p.hidden(l), ref.hidden[l]) < REL_L2, l
        if cycle % 40 == 0 or cycle == 199:
            assert rel_l2(p.logits(), ref.logits) < REL_L2, cycle
        assert rel_l2(p.head_out(), ref.head_out) < REL_L2, cycle
        assert tokens_match(got, ref.tokens, ref.logits), (cycle, got, ref.tokens)
        flip = int(tr.integers(0, G + 1))
        target = S.targets_with_flip(ref.tokens, G, flip, cfg.vocab, tr)
        d = torch.from_numpy(got.astype(np.int32)[None]).cuda()
        t = torch.from_numpy(target[None]).cuda()
        fm.fm_accept_batched(p.h, d, t, k_dev, acc_dev, bonus_dev)
        n_acc, bonus = int(acc_dev.item()), int(bonus_dev.item())
        assert (n_acc, bonus) == accept(got, target, G), cycle
        if np.array_equal(got, ref.tokens):
            same += 1
            assert (n_acc, bonus) == (flip, int(target[flip])), cycle
        p.append(0, S.gen_features(fr, n_acc + 1, cfg.feat_dim), pos)
        pos += n_acc + 1
        anchor = bonus
    assert same >= 190, same
    p.close()


def test_batched_32_sequences_full_shape():
    """The batched serving shape: 32 FlashMap-4B sequences with contexts
    uniform in [512, 8192] (prefilled through the dense path), one batched
    append of acc_i + 1 rows per sequence (acc_i uniform in 0..16), one
    batched 32 x 16-slot draft.  Two sampled sequences (the shortest context
    and a seeded other) are checked against the oracle: tokens, head output
    and logits.  Acceptance of all 32 runs on the device (fm_accept_batched)
    and must equal the acceptance rule bit for bit; for the sampled sequences
    the targets come from the oracle's drafts with a seeded flip."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    from oracle import FlashMap, accept
    n_seqs = 32
    cfg = S.flashmap_4b_config(max_ctx=8192 + 17 + 64, max_seqs=n_seqs)
    w = S.gen_weights(cfg, 1015)
    mod = S.gen_modulation(cfg, 1015)
    rng = S.streams(1015)["workload"]
    L = [int(x) for x in S.batched_lengths(rng, n_seqs)]
    n = [int(x) + 1 for x in rng.integers(0, 17, size=n_seqs)]
    anchors = [int(x) for x in rng.integers(0, cfg.vocab, size=n_seqs)]
    sample = [int(np.argmin(L)), int(rng.integers(0, n_seqs))]
    if sample[1] == sample[0]:
        sample[1] = (sample[0] + 1) % n_seqs
    h = fm.fm_create(cfg, fm.weight_items(w), mod)
    g = torch.Generator(device="cuda")
    g.manual_seed(1015)
    host = {}
    for i in range(n_seqs):
        if i in sample:
            fr = S.streams(1015 + 1 + i)["features"]
            host[i] = (S.gen_features(fr, L[i], cfg.feat_dim), S.gen_features(fr, n[i], cfg.feat_dim))
            f = torch.from_numpy(host[i][0]).cuda()
        else:
            f = torch.randn((L[i], cfg.feat_dim), generator=g, device="cuda")
        fm.fm_context_append(h, i, f, L[i], 0)
        del f
    rows = [torch.from_numpy(host[i][1]).cuda() if i in sample else
            torch.randn((n[i], cfg.feat_dim), generator=g, device="cuda") for i in range(n_seqs)]
    fm.fm_context_append_batched(h, list(range(n_seqs)), torch.cat(rows), n, L)
    pos = [L[i] + n[i] for i in range(n_seqs)]
    tok = torch.zeros((n_seqs, cfg.block), dtype=torch.int32, device="cuda")
    fm.fm_draft(h, list(range(n_seqs)), anchors, pos, tok)
    torch.cuda.synchronize()
    got = tok.cpu().numpy()
    for i in range(n_seqs):
        assert fm.fm_get_length(h, i) == pos[i]
    # the sampled sequences against the oracle (their head output and logits
    # are read before any other draft of the handle)
    o = FlashMap(cfg, {k: t.data for k, t in w.items()}, mod, True)
    refs = {}
    for i in sample:
        st = o.new_state(pos[i] + cfg.block + 2)
        o.context_append(st, host[i][0], 0)
        o.context_append(st, host[i][1], L[i])
        ref = o.draft(st, anchors[i], pos[i])
        refs[i] = ref
        y = np.empty((cfg.block, cfg.target_dim), np.float32)
        fm.fm_debug_copy(h, fm.FM_DEBUG_HEAD_OUT, i, 0, y)
        assert rel_l2(y, ref.head_out) < REL_L2, i
        lg = np.empty((cfg.block, cfg.vocab), np.float32)
        fm.fm_debug_copy(h, fm.FM_DEBUG_LOGITS, i, 0, lg)
        assert rel_l2(lg, ref.logits) < REL_L2, i
        assert tokens_match(got[i], ref.tokens, ref.logits), (i, got[i], ref.tokens)
    # acceptance of every sequence on the device, acceptance counts uniform in 0..16
    tr = S.streams(1015)["tokens"]
    flips = [int(x) for x in tr.integers(0, cfg.block + 1, size=n_seqs)]
    targets = np.stack([S.targets_with_flip(refs[i].tokens if i in refs else got[i], cfg.block, flips[i],
                                            cfg.vocab, tr) for i in range(n_seqs)])
    k = torch.full((n_seqs,), cfg.block, dtype=torch.int32, device="cuda")
    acc = torch.zeros(n_seqs, dtype=torch.int32, device="cuda")
    bonus = torch.zeros(n_seqs, dtype=torch.int32, device="cuda")
    fm.fm_accept_batched(h, tok, torch.from_numpy(targets).cuda(), k, acc, bonus)
    acc, bonus = acc.cpu().numpy(), bonus.cpu().numpy()
    for i in range(n_seqs):
        assert (int(acc[i]), int(bonus[i])) == accept(got[i], targets[i], cfg.block), i
        if i not in refs or np.array_equal(got[i], refs[i].tokens):
            assert int(acc[i]) == flips[i], i
    fm.fm_destroy(h)


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


def test_flashmap_4b_step_persistent(monkeypatch):
    """The opt-in one-launch draft step (FM_PERSISTENT=1: 8-CTA clusters, a
    counter grid barrier between the layer phases) on the FlashMap-4B step:
    the same parity as the launch chain, in at most six launches."""
    monkeypatch.setenv("FM_PERSISTENT", "1")
    cfg = S.flashmap_4b_config()
    p = Pair(cfg, 1002)
    fr = S.streams(1002)["features"]
    p.append(0, S.gen_features(fr, 1024, cfg.feat_dim), 0)
    p.append(0, S.gen_features(fr, 17, cfg.feat_dim), 1024)
    anchor = S.gen_anchor(S.streams(1002)["tokens"], cfg.vocab)
    got, ref = p.draft(0, anchor, 1041)
    assert p.last_launches <= 6, p.last_launches
    for l in range(cfg.n_layers):
        assert rel_l2(p.hidden(l), ref.hidden[l]) < REL_L2, l
    assert rel_l2(p.head_out(), ref.head_out) < REL_L2
    assert tokens_match(got, ref.tokens, ref.logits), (got, ref.tokens)
    p.close()
