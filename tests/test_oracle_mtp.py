"""Pins of the MTP draft head's oracle (ternary_bonsai_2_mtp.js, ``MTPHead.forward``,
``WG_QKPREP``, ``WG_ATTN``, ``MTPRunner``'s draft loop) against a brute-force
scalar restatement, closed forms of NEOX RoPE, and reductions of the graph."""
from __future__ import annotations

import math

import numpy as np
import pytest

import brute
import fm_synth as S
from oracle.mtp import MtpHead, neox_rope


def nano():
    # the smallest head of the same structure: Q8_0 rows need K % 32 == 0
    return S.MtpConfig(hidden=32, inter=64, n_heads=4, n_kv_heads=2, head_dim=16, rot_dims=8, theta=100.0,
                       vocab=64, kv_cap=16)


def raw(w):
    return {n: t.data for n, t in w.items()}


def test_forward_matches_brute_force():
    cfg = nano()
    w = raw(S.gen_mtp_weights(cfg, 21))
    o = MtpHead(cfg, w)
    st = o.new_state()
    rng = S.streams(21)["features"]
    hn = S.gen_mtp_hidden(rng, 3, cfg.hidden)
    # a pass at position 1, then 3 rows at 2..4 over cache rows from 1, then 1 row at 5
    tok = [5, 17, 63]
    kc, vc = [None] * cfg.kv_cap, [None] * cfg.kv_cap
    h1 = S.gen_mtp_hidden(rng, 1, cfg.hidden)
    brute.mtp_forward(w, cfg, [9], h1, 1, 1, kc, vc)
    want = brute.mtp_forward(w, cfg, tok, hn, 2, 1, kc, vc)
    o.forward(st, o.embed([9]), h1.astype(np.float64), 1, 1)
    got = o.forward(st, o.embed(tok), hn.astype(np.float64), 2, 1)
    np.testing.assert_allclose(got.hout, np.array(want), rtol=1e-9, atol=1e-12)
    for p in range(1, 5):
        np.testing.assert_allclose(st.k[p], kc[p], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(st.v[p], vc[p], rtol=1e-9, atol=1e-12)
    h5 = S.gen_mtp_hidden(rng, 1, cfg.hidden)
    want5 = brute.mtp_forward(w, cfg, [40], h5, 5, 1, kc, vc)
    got5 = o.forward(st, o.embed([40]), h5.astype(np.float64), 5, 1)
    np.testing.assert_allclose(got5.hout, np.array(want5), rtol=1e-9, atol=1e-12)


def test_neox_rope_closed_forms():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(16)
    # position 0 is the identity; dims from rot on never move; each pair keeps its length
    np.testing.assert_allclose(neox_rope(x, 0, 8, 100.0), x)
    y = neox_rope(x, 7, 8, 100.0)
    np.testing.assert_array_equal(y[8:], x[8:])
    for i in range(4):
        np.testing.assert_allclose(math.hypot(y[i], y[i + 4]), math.hypot(x[i], x[i + 4]))
    # pair 0 turns by exactly pos radians (frequency theta^0 = 1); pairs are (i, i + rot/2), not (2i, 2i + 1)
    a = 7.0
    np.testing.assert_allclose([y[0], y[4]], [x[0] * math.cos(a) - x[4] * math.sin(a),
                                               x[4] * math.cos(a) + x[0] * math.sin(a)])
    # pair i turns by pos * theta^(-2i/rot): relative positions only in the rotated dot product
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    d1 = neox_rope(q, 11, 8, 100.0)[:8] @ neox_rope(k, 4, 8, 100.0)[:8]
    d2 = neox_rope(q, 27, 8, 100.0)[:8] @ neox_rope(k, 20, 8, 100.0)[:8]
    np.testing.assert_allclose(d1, d2)


def test_single_key_attention_is_the_gated_value_row():
    """With one cached key (kv_lo = pos), softmax is 1: the head's attention
    output is that row's V times sigmoid(gate) per head (kv head h // 2)."""
    cfg = nano()
    w = raw(S.gen_mtp_weights(cfg, 22))
    o = MtpHead(cfg, w)
    st = o.new_state()
    hn = S.gen_mtp_hidden(S.streams(22)["features"], 1, cfg.hidden).astype(np.float64)
    res = o.forward(st, o.embed([3]), hn, 6, 6)
    from oracle.common import rms_norm
    xc = np.concatenate([rms_norm(o.embed([3]), o.w["enorm"], cfg.eps), rms_norm(hn, o.w["hnorm"], cfg.eps)], axis=1)
    a = rms_norm(xc @ o.w["eh_proj"].T, o.w["attn_norm"], cfg.eps)
    qf = (a @ o.w["attn_q"].T)[0]
    v = (a @ o.w["attn_v"].T)[0]
    hd = cfg.head_dim
    for h in range(cfg.n_heads):
        g = h // 2
        gate = qf[h * 2 * hd + hd:(h + 1) * 2 * hd]
        np.testing.assert_allclose(res.gated[0, h * hd:(h + 1) * hd], v[g * hd:(g + 1) * hd] / (1 + np.exp(-gate)))


def test_rows_are_causal_and_passes_compose():
    """Row m attends only to cache rows up to its own position: the first rows
    of a pass do not change when later rows are added, and one pass over four
    rows equals a pass over two then a pass over the other two."""
    cfg = nano()
    w = raw(S.gen_mtp_weights(cfg, 23))
    o = MtpHead(cfg, w)
    hn = S.gen_mtp_hidden(S.streams(23)["features"], 4, cfg.hidden).astype(np.float64)
    tok = [1, 2, 3, 4]
    s1 = o.new_state()
    full = o.forward(s1, o.embed(tok), hn, 3, 3)
    s2 = o.new_state()
    a = o.forward(s2, o.embed(tok[:2]), hn[:2], 3, 3)
    b = o.forward(s2, o.embed(tok[2:]), hn[2:], 5, 3)
    np.testing.assert_allclose(full.hout, np.concatenate([a.hout, b.hout]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s1.k, s2.k)
    np.testing.assert_allclose(s1.v, s2.v)


def test_zero_output_projections_leave_the_projected_input():
    """attn_output = 0 and ffn_down = 0 make the block the identity on
    X = eh_proj [enorm(e) | hnorm(h)]: h' = shared_head_norm(X)."""
    cfg = nano()
    w = raw(S.gen_mtp_weights(cfg, 24))
    for n, k in (("attn_output", cfg.n_heads * cfg.head_dim), ("ffn_down", cfg.inter)):
        w[n] = S.quantize_q8_0(np.zeros((w[n].shape[0], k), np.float32))
    o = MtpHead(cfg, w)
    hn = S.gen_mtp_hidden(S.streams(24)["features"], 2, cfg.hidden).astype(np.float64)
    res = o.forward(o.new_state(), o.embed([7, 8]), hn, 0, 0)
    from oracle.common import rms_norm
    xc = np.concatenate([rms_norm(o.embed([7, 8]), o.w["enorm"], cfg.eps), rms_norm(hn, o.w["hnorm"], cfg.eps)], axis=1)
    x = xc @ o.w["eh_proj"].T
    np.testing.assert_allclose(res.hout, rms_norm(x, o.w["shared_head_norm"], cfg.eps))


def test_draft_chains_the_head():
    """A depth-d draft is one pass over the pending rows and d - 1 single-row
    passes on the previous draft and h'; its first tokens do not depend on d."""
    cfg = nano()
    w = raw(S.gen_mtp_weights(cfg, 25))
    o = MtpHead(cfg, w)
    hn = S.gen_mtp_hidden(S.streams(25)["features"], 2, cfg.hidden).astype(np.float64)
    d3, lg3, h3 = o.draft(o.new_state(), [11, 12], hn, 4, 2, 3)
    d1, lg1, _ = o.draft(o.new_state(), [11, 12], hn, 4, 2, 1)
    assert d3[0] == d1[0] and len(d3) == 3
    np.testing.assert_allclose(lg3[0], lg1[0])
    for k in range(3):
        assert d3[k] == int(np.argmax(lg3[k]))
    # step 2 by hand: the first draft at position 6 with the last row's h'
    st = o.new_state()
    r0 = o.forward(st, o.embed([11, 12]), hn, 4, 2)
    r1 = o.forward(st, o.embed([int(d3[0])]), r0.hout[-1:], 6, 2)
    np.testing.assert_allclose(lg3[1], o.logits(r1.hout)[0])
