"""Parity of the CUDA path (through the C ABI) with the oracle on small
workloads that span several tiles and ragged tails: the tiny FlashMap-shaped
drafter (both table formats), a small DFlash drafter, ragged append sizes,
rewinds, the empty-context draft, and acceptance."""
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


def small_dflash(**kw):
    c = S.DrafterConfig(S.VARIANT_DFLASH, dim=256, n_heads=2, head_dim=128, n_layers=2, ff_dim=512, block=5,
                        target_dim=320, n_taps=2, vocab=4096, lm_format=S.LM_BF16, max_ctx=160)
    return c.replace(**kw)


def check_draft(p: Pair, got, ref, layers=True):
    if layers:
        for l in range(p.cfg.n_layers):
            e = rel_l2(p.hidden(l), ref.hidden[l])
            assert e < REL_L2, (l, e)
    e = rel_l2(p.head_out(), ref.head_out)
    assert e < REL_L2, e
    lg = p.logits()
    e = rel_l2(lg, ref.logits)
    assert e < REL_L2, e
    assert tokens_match(got, ref.tokens, ref.logits), (got, ref.tokens)
    # the fused argmax agrees with the argmax of the recomputed logits
    assert np.array_equal(got, np.argmax(lg, axis=-1))


def check_cache(p: Pair, seq, rows):
    st = p.state(seq)
    for l in range(p.cfg.n_layers):
        for which, ref in (("k", st.k[l]), ("v", st.v[l])):
            got = p.cache(seq, l, which)[:rows]
            want = ref[:rows]
            assert rel_l2(got, want) < 1e-3, (l, which, rel_l2(got, want))
            # the f16 store matches the oracle's f16 rounding up to one step of the
            # element plus a small fraction of the row's scale (f32 vs f64 before rounding)
            rms = np.sqrt(np.mean(want.astype(np.float64) ** 2, axis=1, keepdims=True))
            step = np.abs(want) * 2.0 ** -10 + 1e-4 * rms + 2.0 ** -24
            bad = np.abs(got - want) > step
            assert not bad.any(), (l, which, int(bad.sum()), float(np.abs(got - want)[bad].max()))


@pytest.mark.parametrize("lm", [S.LM_BF16, S.LM_Q8_0])
def test_tiny_flashmap_one_step(lm):
    cfg = S.tiny_config(max_ctx=128).replace(lm_format=lm)
    p = Pair(cfg, 1001)
    rng = S.streams(1001)["features"]
    p.append(0, S.gen_features(rng, 64, cfg.feat_dim), 0)
    check_cache(p, 0, 64)
    anchor = S.gen_anchor(S.streams(1001)["tokens"], cfg.vocab)
    got, ref = p.draft(0, anchor, 64)
    if persistent_step_requested():
        assert p.last_launches <= 6, p.last_launches      # anchor, K/V, the step, the lm_head
    check_draft(p, got, ref)
    check_cache(p, 0, 65)
    p.close()


@pytest.mark.parametrize("target_dim", [384, 512])
def test_tiny_flashmap_q8_chunk_pairs(target_dim):
    """Q8_0 lm_head widths whose 64-column chunk count per tile is 6 (pairs, one
    MMA issuer) and 8 (pairs alternating between two issuers)."""
    cfg = S.tiny_config(max_ctx=96).replace(lm_format=S.LM_Q8_0, target_dim=target_dim)
    p = Pair(cfg, 1005)
    p.append(0, S.gen_features(S.streams(1005)["features"], 40, cfg.feat_dim), 0)
    got, ref = p.draft(0, 123, 40)
    check_draft(p, got, ref)
    p.close()


def test_tiny_flashmap_ragged_appends_and_rewind():
    cfg = S.tiny_config(max_ctx=160)
    p = Pair(cfg, 1002)
    rng = S.streams(1002)["features"]
    feats = S.gen_features(rng, 120, cfg.feat_dim)
    start = 0
    for n in (1, 5, 16, 17, 31, 32, 18):   # 120 rows in ragged pieces (33-row pieces below)
        p.append(0, feats[start:start + n], start)
        start += n
    check_cache(p, 0, 120)
    k_before = [p.cache(0, l, "k").copy() for l in range(cfg.n_layers)]
    # rewind to 100 and re-append the same rows: bit-identical cache
    p.append(0, feats[100:120], 100)
    for l in range(cfg.n_layers):
        assert np.array_equal(p.cache(0, l, "k")[:120], k_before[l][:120])
    got, ref = p.draft(0, 7, 120)
    check_draft(p, got, ref)
    p.close()


def test_tiny_flashmap_long_append_crosses_chunks():
    cfg = S.tiny_config(max_ctx=160)
    p = Pair(cfg, 1003)
    feats = S.gen_features(S.streams(1003)["features"], 97, cfg.feat_dim)
    p.append(0, feats, 0)                    # 97 rows: three 32-row passes and a tail
    check_cache(p, 0, 97)
    got, ref = p.draft(0, 4095, 97)
    check_draft(p, got, ref)
    p.close()


def test_tiny_flashmap_empty_context_draft():
    cfg = S.tiny_config(max_ctx=64)
    p = Pair(cfg, 1004)
    got, ref = p.draft(0, 11, 0)             # cross keys = the anchor slot alone
    check_draft(p, got, ref)
    check_cache(p, 0, 1)
    p.close()


def test_tiny_flashmap_draft_accept_cycles():
    """Several verify rounds: draft, targets with a seeded flip, accept on host
    and device, append acc + 1 fresh rows from the anchor slot."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    from oracle import accept
    cfg = S.tiny_config(max_ctx=200)
    p = Pair(cfg, 1005)
    fr = S.streams(1005)["features"]
    tr = S.streams(1005)["tokens"]
    p.append(0, S.gen_features(fr, 40, cfg.feat_dim), 0)
    pos, anchor = 40, 3
    for cycle in range(6):
        got, ref = p.draft(0, anchor, pos)
        check_draft(p, got, ref, layers=(cycle == 0))
        flip = int(tr.integers(0, cfg.block + 1))
        target = S.targets_with_flip(ref.tokens, cfg.block, flip, cfg.vocab, tr)
        want = accept(ref.tokens, target, cfg.block)
        assert fm.fm_accept(ref.tokens.astype(np.int32), target, cfg.block) == want
        d = torch.from_numpy(ref.tokens.astype(np.int32)[None]).cuda()
        t = torch.from_numpy(target[None]).cuda()
        k = torch.full((1,), cfg.block, dtype=torch.int32, device="cuda")
        acc = torch.zeros(1, dtype=torch.int32, device="cuda")
        bonus = torch.zeros(1, dtype=torch.int32, device="cuda")
        fm.fm_accept_batched(p.h, d, t, k, acc, bonus)
        assert (int(acc.item()), int(bonus.item())) == want
        n = want[0] + 1
        p.append(0, S.gen_features(fr, n, cfg.feat_dim), pos)
        pos += n
        anchor = want[1]
    check_cache(p, 0, pos)
    p.close()


def test_small_dflash_steps():
    cfg = small_dflash()
    p = Pair(cfg, 1006)
    fr = S.streams(1006)["features"]
    p.append(0, S.gen_features(fr, 70, cfg.feat_dim), 0)
    got, ref = p.draft(0, 17, 70)
    check_draft(p, got, ref)
    # verify cycle: append acc + 1 rows at the anchor position, draft again
    p.append(0, S.gen_features(fr, 3, cfg.feat_dim), 70)
    got, ref = p.draft(0, 99, 73)
    check_draft(p, got, ref)
    p.close()


def test_small_dflash_long_context_sharp_scores():
    """Attention with head dim 128 over 32,768 context rows, with the query and
    key projections scaled up so that scores spread over tens of log2 units:
    each key range holds eight 128-key tiles, and later tiles often beat the
    first tile's maximum by more than 2^8, which moves the range's softmax
    reference and rescales its accumulator.  Hidden states, head output and
    logits against the oracle."""
    cfg = small_dflash(max_ctx=32768 + 16)

    def sharpen(w):
        for l in range(cfg.n_layers):
            for n in ("q", "k"):
                t = w[f"bb.{l}.{n}"]
                t.data = S.f32_to_bf16_bits(S.bf16_bits_to_f32(t.data) * 16.0)
    p = Pair(cfg, 1009, edit=sharpen)
    fr = S.streams(1009)["features"]
    for start in range(0, 32768, 4096):
        p.append(0, S.gen_features(fr, 4096, cfg.feat_dim), start)
    got, ref = p.draft(0, 21, 32768)
    check_draft(p, got, ref)
    p.close()


def test_small_dflash_empty_context():
    cfg = small_dflash()
    p = Pair(cfg, 1007)
    got, ref = p.draft(0, 5, 0)              # attention over the block alone
    check_draft(p, got, ref)
    p.close()


def test_errors_are_reported_not_raised_on_device():
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.tiny_config(max_ctx=64)
    p = Pair(cfg, 1008, keep_hidden=False)
    feats = S.gen_features(S.streams(1008)["features"], 8, cfg.feat_dim)
    with pytest.raises(fm.FmError) as e:
        p.append(0, feats, 3, oracle=False)           # start beyond the length
    assert e.value.status == fm.FM_ERR_STATE
    with pytest.raises(fm.FmError) as e:
        p.append(0, S.gen_features(S.streams(1)["features"], 60, cfg.feat_dim), 0, oracle=False)
    assert e.value.status == fm.FM_ERR_CONTEXT_FULL
    with pytest.raises(fm.FmError) as e:
        p.draft(0, cfg.vocab, 0, oracle=False)        # anchor out of range
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    with pytest.raises(fm.FmError) as e:
        p.draft(0, 1, 5, oracle=False)                # pos != length
    assert e.value.status == fm.FM_ERR_STATE
    with pytest.raises(fm.FmError) as e:
        p.append(1, feats, 0, oracle=False)           # seq beyond max_seqs
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    p.close()


def test_tiny_flashmap_dense_prefill_tcgen05():
    """Appends of >= 128 rows run the tcgen05 GEMMs (f16 operands): cache rows
    and the draft that reads them stay within the parity bars."""
    cfg = S.tiny_config(max_ctx=640)
    p = Pair(cfg, 1009)
    feats = S.gen_features(S.streams(1009)["features"], 600, cfg.feat_dim)
    p.append(0, feats[:300], 0)             # one dense pass with a ragged last M tile (300 = 2 * 128 + 44)
    p.append(0, feats[300:557], 300)        # a second pass that starts mid-context
    st = p.state(0)
    for l in range(cfg.n_layers):
        for which, want in (("k", st.k[l]), ("v", st.v[l])):
            got = p.cache(0, l, which)[:557]
            assert rel_l2(got, want[:557]) < 1e-3, (l, which, rel_l2(got, want[:557]))
    got, ref = p.draft(0, 123, 557)
    check_draft(p, got, ref)
    p.close()


def test_tiny_flashmap_batched_sequences():
    """Several independent sequences with ragged lengths: one batched append
    and one batched draft match the oracle run per sequence."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.tiny_config(max_ctx=200).replace(max_seqs=4)
    p = Pair(cfg, 1010)
    fr = S.streams(1010)["features"]
    lens = [5, 64, 37, 130]
    for s, n in enumerate(lens):
        p.append(s, S.gen_features(fr, n, cfg.feat_dim), 0)
    # batched append of acc + 1 rows per sequence (rows concatenated in sequence order)
    extra = [1, 17, 3, 9]
    rows = [S.gen_features(fr, n, cfg.feat_dim) for n in extra]
    feats = torch.from_numpy(np.concatenate(rows)).cuda()
    ids = [2, 0, 3, 1]
    fm.fm_context_append_batched(p.h, ids, feats, [extra[0], extra[1], extra[2], extra[3]],
                                 [lens[i] for i in ids])
    for j, s in enumerate(ids):
        p.oracle.context_append(p.state(s), rows[j], lens[s])
    pos = [lens[s] + extra[ids.index(s)] for s in range(4)]
    anchors = [11, 22, 33, 44]
    tok = torch.zeros((4, cfg.block), dtype=torch.int32, device="cuda")
    fm.fm_draft(p.h, [0, 1, 2, 3], anchors, pos, tok)
    torch.cuda.synchronize()
    got = tok.cpu().numpy()
    for s in range(4):
        ref = p.oracle.draft(p.state(s), anchors[s], pos[s])
        assert tokens_match(got[s], ref.tokens, ref.logits), (s, got[s], ref.tokens)
        assert fm.fm_get_length(p.h, s) == pos[s]
    p.close()


def test_tiny_flashmap_large_dc_offset():
    """A residual stream far from zero mean: x_embed's bias set to 1000 makes
    h0 ~ 1000 + O(0.4), so every LayerNorm sees |mean| / std ~ 2500.  The
    variance must come from deviations about the mean (the page's two-pass
    lnMod); a variance formed as E[x^2] - mean^2 in f32 loses every digit of it
    (mean^2 ~ 1e6, f32 spacing ~0.06, variance ~0.15) and fails the bars."""
    def offset(w):
        t = w["x_embed.bias"]
        t.data = S.f32_to_bf16_bits(np.full(t.shape, 1000.0, np.float32))
    cfg = S.tiny_config(max_ctx=96)
    p = Pair(cfg, 1011, edit=offset)
    assert abs(float(p.oracle.h0.mean())) > 900.0 and float(p.oracle.h0.std()) < 1.0
    p.append(0, S.gen_features(S.streams(1011)["features"], 40, cfg.feat_dim), 0)
    got, ref = p.draft(0, 321, 40)
    check_draft(p, got, ref)
    p.close()


@pytest.mark.parametrize("lm", [S.LM_BF16, S.LM_Q8_0])
def test_argmax_ties_go_to_the_lowest_index(lm):
    """Every odd table row is a copy of the even row before it, so each slot's
    best logit is tied between rows 2j and 2j + 1: the fused two-pass argmax
    must return the even (lower) index, as numpy's first-occurrence argmax
    does; identical rows give bit-identical logits on the device."""
    def pairs(w):
        t = w["token_embd.weight"]
        t.data = t.data.copy()
        t.data[1::2] = t.data[0::2]
    cfg = S.tiny_config(max_ctx=96).replace(lm_format=lm)
    p = Pair(cfg, 1012, edit=pairs)
    p.append(0, S.gen_features(S.streams(1012)["features"], 40, cfg.feat_dim), 0)
    got, ref = p.draft(0, 200, 40)
    lg = p.logits()
    assert np.array_equal(lg[:, 0::2], lg[:, 1::2])          # the ties are exact on the device
    assert np.all(got % 2 == 0), got
    assert np.array_equal(got, np.argmax(lg, axis=-1))
    # against the oracle where the winning pair is clear of every other row
    best = ref.tokens
    rest = ref.logits.copy()
    rows = np.arange(cfg.block)
    rest[rows, best] = -np.inf
    rest[rows, best + 1] = -np.inf
    clear = ref.logits[rows, best] - rest.max(axis=1) >= 1e-3
    assert np.all(best % 2 == 0)
    assert np.array_equal(got[clear], best[clear]), (got, best)
    assert rel_l2(lg, ref.logits) < REL_L2
    p.close()


def test_allocation_failure_is_reported_and_released():
    """FM_FAULT_INJECT=alloc:N makes the N-th device allocation of fm_create
    fail (a host-side fault, nothing on the GPU faults): fm_create returns
    FM_ERR_OOM with a reason, frees what it had allocated, and a later
    fm_create on the same device works."""
    import os
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.tiny_config(max_ctx=96)
    w = S.gen_weights(cfg, 1013)
    mod = S.gen_modulation(cfg, 1013)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        for n in (1, 7, 40):
            os.environ["FM_FAULT_INJECT"] = f"alloc:{n}"
            with pytest.raises(fm.FmError) as e:
                fm.fm_create(cfg, fm.weight_items(w), mod)
            assert e.value.status == fm.FM_ERR_OOM
            assert f"allocation {n}" in str(e.value)
    finally:
        os.environ.pop("FM_FAULT_INJECT", None)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (16 << 20)   # nothing of the failed handles is kept
    h = fm.fm_create(cfg, fm.weight_items(w), mod)
    tok = torch.zeros((1, cfg.block), dtype=torch.int32, device="cuda")
    fm.fm_draft(h, [0], [9], [0], tok)
    fm.fm_synchronize(h)
    fm.fm_destroy(h)


def test_bounded_wait_gives_up_and_is_reported():
    """A device wait that can never complete (an mbarrier phase nothing
    completes) gives up after its budget, raises the handle's error word and
    returns: fm_synchronize reports FM_ERR_TIMEOUT once, and the handle keeps
    drafting correctly afterwards."""
    import time
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.tiny_config(max_ctx=96)
    p = Pair(cfg, 1014)
    p.append(0, S.gen_features(S.streams(1014)["features"], 30, cfg.feat_dim), 0)
    fm.fm_synchronize(p.h)
    t0 = time.perf_counter()
    fm.fm_selftest_wait_timeout(p.h, 20000)          # 20 ms budget
    with pytest.raises(fm.FmError) as e:
        fm.fm_synchronize(p.h)
    assert e.value.status == fm.FM_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    fm.fm_synchronize(p.h)                           # reported once, then cleared
    got, ref = p.draft(0, 77, 30)
    check_draft(p, got, ref)
    fm.fm_synchronize(p.h)
    p.close()


def test_time_conditioning_table_and_draft():
    """fm_time_conditioning builds the adaLN table of the jump 0 -> 1 from the
    time-conditioning linears on the device; the table matches the oracle's,
    and a drafter created from it drafts what the oracle drafts from the
    oracle's own table."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    from oracle import FlashMap
    from oracle.timecond import time_conditioning
    cfg = S.tiny_config(max_ctx=96)
    w = S.gen_weights(cfg, 1016)
    tw = S.gen_time_cond_weights(cfg, 1016, time_dim=256, cond_dim=256)
    table = torch.full(((3 * cfg.n_layers + 1) * 3 * cfg.dim,), float("nan"), device="cuda")
    # the whole checkpoint list: the entry point picks the tensors it needs
    fm.fm_time_conditioning(cfg, fm.weight_items({**w, **tw}), 256, 256, 1000.0, 0.0, 1.0, table)
    want = time_conditioning({n: t.data for n, t in tw.items()}, cfg.n_layers, cfg.dim, 256, 1000.0, 0.0, 1.0)
    got = table.cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, want) < 1e-5, rel_l2(got, want)
    h = fm.fm_create(cfg, fm.weight_items(w), table)
    o = FlashMap(cfg, {n: t.data for n, t in w.items()}, want, False)
    st = o.new_state()
    feats = S.gen_features(S.streams(1016)["features"], 30, cfg.feat_dim)
    fm.fm_context_append(h, 0, torch.from_numpy(feats).cuda(), 30, 0)
    o.context_append(st, feats, 0)
    tok = torch.zeros((1, cfg.block), dtype=torch.int32, device="cuda")
    fm.fm_draft(h, [0], [55], [30], tok)
    torch.cuda.synchronize()
    ref = o.draft(st, 55, 30)
    y = np.empty((cfg.block, cfg.target_dim), np.float32)
    fm.fm_debug_copy(h, fm.FM_DEBUG_HEAD_OUT, 0, 0, y)
    assert rel_l2(y, ref.head_out) < REL_L2
    assert tokens_match(tok.cpu().numpy()[0], ref.tokens, ref.logits)
    fm.fm_destroy(h)
    # a missing linear is reported, nothing is written
    with pytest.raises(fm.FmError) as e:
        fm.fm_time_conditioning(cfg, fm.weight_items({k: v for k, v in tw.items() if "final_adaln" not in k}),
                                256, 256, 1000.0, 0.0, 1.0, table)
    assert e.value.status == fm.FM_ERR_INVALID_ARG
