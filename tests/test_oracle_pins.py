"""Pins of the CPU oracle against things other than itself: closed forms,
invariants, independent library routines, the pages' printed constants and
brute force on micro dims.  CPU only (no GPU marker)."""
from __future__ import annotations

import itertools
import json
import math
import os
import struct

import numpy as np
import pytest
import scipy.stats
import torch

import brute
import fm_synth as S
from oracle import DFlash, FlashMap, accept
from oracle import common as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def micro_flashmap(lm_format=S.LM_Q8_0, **kw):
    c = S.DrafterConfig(S.VARIANT_FLASHMAP, dim=8, n_heads=2, head_dim=4, n_layers=2, ff_dim=12, block=4,
                        target_dim=32, n_taps=2, vocab=16, lm_format=lm_format, max_ctx=24)
    return c.replace(**kw)


def micro_dflash(**kw):
    c = S.DrafterConfig(S.VARIANT_DFLASH, dim=8, n_heads=2, head_dim=4, n_layers=2, ff_dim=16, block=3,
                        target_dim=8, n_taps=2, vocab=16, lm_format=S.LM_BF16, max_ctx=24)
    return c.replace(**kw)


def raw_weights(cfg, seed):
    return {n: t.data for n, t in S.gen_weights(cfg, seed).items()}


# ---------------------------------------------------------------- formats

def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]      # drop inf/nan patterns
    want = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(C.bf16_to_f64(bits), want)
    assert C.bf16_to_f64(np.array([0x3F80, 0xC000, 0x3F81], np.uint16)).tolist() == [1.0, -2.0, 1.0 + 2 ** -7]


def test_f16_store_matches_struct_half():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(2000) * np.exp(rng.uniform(-12, 8, 2000))
    want = [struct.unpack("<e", struct.pack("<e", float(v)))[0] for v in x]
    np.testing.assert_array_equal(C.f16_store(x), want)


def test_q8_0_dequant_against_byte_parsing():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 64)).astype(np.float32) * 0.02
    raw = S.quantize_q8_0(x)
    got = C.q8_0_dequant(raw, 64)
    for r in range(5):
        np.testing.assert_array_equal(got[r], brute.q8_row(raw[r], 64))
    # hand-built block: scale 0.5 (f16 0x3800) then q = 1, -2, 127, -128, 0, ...
    blk = bytearray(struct.pack("<H", 0x3800)) + struct.pack("32b", 1, -2, 127, -128, *([0] * 28))
    v = C.q8_0_dequant(np.frombuffer(bytes(blk), np.uint8)[None, :], 32)[0]
    assert v[:5].tolist() == [0.5, -1.0, 63.5, -64.0, 0.0]
    # the quantiser the generator uses reconstructs within half a step
    step = np.abs(x.reshape(5, 2, 32)).max(-1) / 127
    err = np.abs(got - x).reshape(5, 2, 32).max(-1)
    assert np.all(err <= step * 0.5 + 1e-3 * step + 1e-12)


# ---------------------------------------------------------------- primitives

def test_linear_is_out_in_layout():
    rng = np.random.default_rng(3)
    W = rng.standard_normal((3, 5))
    b = rng.standard_normal(3)
    x = rng.standard_normal((2, 5))
    got = C.linear(x, W, b)
    for t in range(2):
        np.testing.assert_allclose(got[t], brute.matvec(W.tolist(), x[t].tolist(), b.tolist()), rtol=1e-14)


def test_rms_norm_closed_forms():
    w = np.array([1.0, 2.0, -3.0, 0.5])
    for c, eps in [(2.0, 1e-6), (0.1, 1e-5), (7.0, 0.0)]:
        got = C.rms_norm(np.full((1, 4), c), w, eps)[0]
        np.testing.assert_allclose(got, w * c / math.sqrt(c * c + eps), rtol=1e-15)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 16))
    y = C.rms_norm(x, np.ones(16), 0.0)
    np.testing.assert_allclose((y * y).mean(-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(C.rms_norm(5.0 * x, np.ones(16), 0.0), y, rtol=1e-14)


def test_layer_norm_modulate_closed_forms():
    n = 6
    sc = np.linspace(-0.3, 0.4, n)
    sh = np.linspace(1.0, -1.0, n)
    # a constant row normalises to zero, leaving the shift
    np.testing.assert_array_equal(C.layer_norm_modulate(np.full((1, n), 3.25), sc, sh, 1e-6)[0], sh)
    # [a, -a]: mean 0, population variance a^2
    a, eps = 0.7, 1e-3
    got = C.layer_norm_modulate(np.array([[a, -a]]), np.zeros(2), np.zeros(2), eps)[0]
    np.testing.assert_allclose(got, np.array([a, -a]) / math.sqrt(a * a + eps), rtol=1e-15)
    # eps = 0: zero mean, sum of squares = n (divide by n, not n - 1)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 10)) + 3.0
    y = C.layer_norm_modulate(x, np.zeros(10), np.zeros(10), 0.0)
    np.testing.assert_allclose(y.sum(-1), 0.0, atol=1e-12)
    np.testing.assert_allclose((y * y).sum(-1), 10.0, rtol=1e-13)
    # modulation acts as (1 + scale) * z + shift
    y2 = C.layer_norm_modulate(x, np.full(10, 0.5), np.full(10, -2.0), 0.0)
    np.testing.assert_allclose(y2, 1.5 * y - 2.0, rtol=1e-13)


def test_head_norm_weight_indexed_by_channel():
    x = np.array([[1.0, 0, 0, 0, 0, 2.0, 0, 0]])
    w = np.array([1.0, 2.0, 3.0, 4.0])
    got = C.head_rms_norm(x, w, 0.0, 4)[0]
    # head 0: rms = 1/2 -> [2, 0, 0, 0]; head 1: rms = 1 -> [0, 4, 0, 0]
    np.testing.assert_allclose(got, [2.0, 0, 0, 0, 0, 4.0, 0, 0], rtol=1e-15)


def test_rope_closed_form_interleaved_pairs():
    hd, theta, p = 4, 100.0, 3
    x = np.array([[1.0, 2.0, -0.5, 0.25]])
    got = C.rope_interleaved(x, np.array([p]), hd, theta)[0]
    a0, a1 = 3.0, 3.0 * 100.0 ** -0.5        # pair 0 turns by p, pair 1 by p * theta^(-2/hd)
    want = [1.0 * math.cos(a0) - 2.0 * math.sin(a0), 2.0 * math.cos(a0) + 1.0 * math.sin(a0),
            -0.5 * math.cos(a1) - 0.25 * math.sin(a1), 0.25 * math.cos(a1) - 0.5 * math.sin(a1)]
    np.testing.assert_allclose(got, want, rtol=1e-14)


def test_rope_invariants():
    rng = np.random.default_rng(6)
    hd, theta = 128, 1e4
    q = rng.standard_normal((1, 2 * hd))
    k = rng.standard_normal((1, 2 * hd))
    np.testing.assert_array_equal(C.rope_interleaved(q, np.array([0]), hd, theta), q)
    for p in (1, 1041, 32768):
        r = C.rope_interleaved(q, np.array([p]), hd, theta)
        np.testing.assert_allclose(np.linalg.norm(r.reshape(2, hd), axis=1),
                                   np.linalg.norm(q.reshape(2, hd), axis=1), rtol=1e-13)
    # <R(p) q, R(s) k> depends only on p - s
    d1 = C.rope_interleaved(q, np.array([20]), hd, theta) @ C.rope_interleaved(k, np.array([5]), hd, theta).T
    d2 = C.rope_interleaved(q, np.array([27]), hd, theta) @ C.rope_interleaved(k, np.array([12]), hd, theta).T
    np.testing.assert_allclose(d1, d2, rtol=1e-11)


def test_attention_invariants_and_brute_force():
    rng = np.random.default_rng(7)
    hd, h = 4, 2
    q = rng.standard_normal((3, h * hd))
    k = rng.standard_normal((5, h * hd))
    v = rng.standard_normal((5, h * hd))
    np.testing.assert_allclose(C.attention(q, k, v, hd), brute.attend(q.tolist(), k.tolist(), v.tolist(), hd),
                               rtol=1e-13)
    # one key returns its value row exactly
    np.testing.assert_allclose(C.attention(q, k[:1], v[:1], hd), np.tile(v[:1], (3, 1)), rtol=1e-15)
    # constant values: weights sum to one
    np.testing.assert_allclose(C.attention(q, k, np.full((5, h * hd), 2.5), hd), 2.5, rtol=1e-14)
    # identical keys: the mean of the values
    np.testing.assert_allclose(C.attention(q, np.tile(k[:1], (5, 1)), v, hd), np.tile(v.mean(0), (3, 1)),
                               rtol=1e-13)
    # a key far ahead of the others takes all the weight
    kk = k.copy()
    kk[2] = q[0] * 1e3
    np.testing.assert_allclose(C.attention(q[:1], kk, v, hd), v[2:3], rtol=1e-12)


def test_gelu_against_libm_and_normal_cdf():
    xs = np.linspace(-8, 8, 801)
    got = C.gelu_erf(xs)
    np.testing.assert_allclose(got, [0.5 * x * (1 + math.erf(x / math.sqrt(2))) for x in xs], rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(got, xs * scipy.stats.norm.cdf(xs), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(got - C.gelu_erf(-xs), xs, atol=1e-13)


def test_gelu_within_the_pages_erf_bound():
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))["erf_approximation"]
    p, a, bound = g["p"], g["a"], g["abs_error_bound"]

    def erf_as(z):
        s = 1.0 if z >= 0 else -1.0
        t = 1.0 / (1.0 + p * abs(z))
        poly = ((((a[4] * t + a[3]) * t + a[2]) * t + a[1]) * t + a[0]) * t
        return s * (1.0 - poly * math.exp(-z * z))

    xs = np.linspace(-6, 6, 1201)
    approx = np.array([0.5 * x * (1 + erf_as(x / math.sqrt(2))) for x in xs])
    assert np.all(np.abs(approx - C.gelu_erf(xs)) <= 0.5 * np.abs(xs) * bound + 1e-15)


def test_gelu_tanh_pins():
    xs = np.linspace(-6, 6, 601)
    got = C.gelu_tanh(xs)
    np.testing.assert_allclose(got - C.gelu_tanh(-xs), xs, atol=1e-13)
    u = math.sqrt(2 / math.pi) * (1 + 0.044715)
    assert abs(C.gelu_tanh(np.array([1.0]))[0] - 0.5 * (1 + math.tanh(u))) < 1e-15
    assert np.max(np.abs(got - C.gelu_erf(xs))) < 1e-3
    assert C.gelu_tanh(np.array([0.0]))[0] == 0.0


def test_argmax_ties_go_to_lowest_index():
    r = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 3.0, 3.0, 3.0]])
    assert C.argmax_rows(r).tolist() == [1, 0]
    assert C.top2_margin(r).tolist() == [0.0, 0.0]


def test_top2_margin_against_brute_force():
    """The gap between the best and the runner-up logit of each row, against a
    sort written out by hand on small rows: hand-made cases (a clear winner, a
    tie, negatives, a duplicate runner-up) and seeded random rows."""
    cases = np.array([[1.0, 4.0, 2.5, -3.0], [-1.0, -5.0, -2.0, -1.5], [7.0, 7.0, 1.0, 0.0],
                      [0.0, 2.0, 9.0, 2.0]])
    assert C.top2_margin(cases).tolist() == [1.5, 0.5, 0.0, 7.0]
    rng = np.random.default_rng(31)
    rows = rng.standard_normal((50, 7))
    for row, m in zip(rows, C.top2_margin(rows)):
        vals = list(row)
        best = max(vals)
        vals.remove(best)   # one copy: a tied runner-up gives 0
        assert m == best - max(vals)


def test_accept_brute_force():
    k, V = 4, 3
    for d in itertools.product(range(V), repeat=k):
        for t in itertools.product(range(V), repeat=k + 1):
            acc, bonus = accept(d, t, k)
            want = next((i for i in range(k) if d[i] != t[i]), k)
            assert (acc, bonus) == (want, t[want])
    rng = np.random.default_rng(8)
    for flip in range(17):
        drafts = rng.integers(0, 1000, 16)
        t = S.targets_with_flip(drafts, 16, flip, 1000, rng)
        assert accept(drafts, t, 16)[0] == flip
    assert accept([5, 6], [5, 6, 9], 0) == (0, 5)


def test_page_constants_in_workload_configs():
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    c = S.flashmap_4b_config()
    f = g["flashmap_cfg"]
    assert (c.dim, c.n_heads, c.head_dim, c.n_layers, c.ff_dim, c.block, c.target_dim) == \
        (f["dim"], f["heads"], f["hd"], f["layers"], f["ff"], f["block"], f["targetDim"])
    assert (c.rope_theta, c.ln_eps, c.rms_eps, c.qk_eps) == (f["theta"], f["lnEps"], f["rmsEps"], f["qkEps"])
    assert c.feat_dim == g["flashmap_tapped_layers"]["feature_width"] == \
        len(g["flashmap_tapped_layers"]["layers"]) * c.target_dim
    d = S.dflash_config()
    dd = g["dflash_defaults"]
    assert (d.block, d.dim, d.n_layers, d.n_heads, d.ff_dim // d.dim, d.n_taps) == \
        (dd["gamma"], dd["dDraft"], dd["nLayers"], dd["nHeads"], dd["ffMult"], dd["n_taps"])
    assert S.quantize_q8_0(np.zeros((1, 32), np.float32)).shape[1] == g["q8_0_block"]["bytes_per_block"]


# ---------------------------------------------------------------- composed forward

@pytest.mark.parametrize("lm", [S.LM_Q8_0, S.LM_BF16])
def test_flashmap_matches_brute_force(lm):
    cfg = micro_flashmap(lm)
    w = raw_weights(cfg, 11)
    mod = S.gen_modulation(cfg, 11)
    rng = S.streams(11)["features"]
    feats = S.gen_features(rng, 5, cfg.feat_dim)
    o = FlashMap(cfg, w, mod, lm == S.LM_Q8_0)
    b = brute.BruteFlashMap(cfg, w, mod, lm == S.LM_Q8_0)
    np.testing.assert_allclose(o.h0, b.h0, rtol=1e-12)
    st = o.new_state()
    o.context_append(st, feats, 0)
    b.append(feats, 0)
    r = o.draft(st, 7, 5)
    toks, logits, Y, hidden = b.draft(7, 5)
    for l in range(cfg.n_layers):
        for p in range(6):
            np.testing.assert_allclose(st.k[l][p], b.K[l][p], rtol=1e-6, atol=1e-9)
            np.testing.assert_allclose(st.v[l][p], b.V[l][p], rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(r.hidden[l], hidden[l], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(r.head_out, Y, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(r.logits, logits, rtol=1e-9, atol=1e-12)
    assert r.tokens.tolist() == toks


def test_flashmap_zero_gates_reduce_to_h0():
    cfg = micro_flashmap()
    w = raw_weights(cfg, 12)
    mod = S.gen_modulation(cfg, 12).astype(np.float64).reshape(-1, 3, cfg.dim)
    mod[:, 2, :] = 0.0                        # every gate zero
    o = FlashMap(cfg, w, mod.reshape(-1), True)
    st = o.new_state()
    o.context_append(st, S.gen_features(S.streams(12)["features"], 3, cfg.feat_dim), 0)
    r = o.draft(st, 3, 3)
    for h in r.hidden:
        np.testing.assert_array_equal(h, np.tile(o.h0, (cfg.block, 1)))
    # closed form of the output: final adaLN of h0, head, E
    E = C.q8_0_dequant(w["token_embd.weight"], cfg.target_dim)
    fin = mod[-1]
    z = (o.h0 - o.h0.mean()) / np.sqrt(o.h0.var() + cfg.ln_eps) * (1 + fin[0]) + fin[1]
    y = C.bf16_to_f64(w["head.weight"]) @ z + C.bf16_to_f64(w["head.bias"])
    assert len(set(r.tokens.tolist())) == 1
    assert r.tokens[0] == int(np.argmax(E @ y))


def test_flashmap_layer0_self_attention_returns_v_row():
    """All slots start at h0, so every slot's self-attention output at layer 0
    is the shared value row whatever q, k and RoPE are."""
    cfg = micro_flashmap(n_layers=1)
    w = raw_weights(cfg, 13)
    mod = S.gen_modulation(cfg, 13).astype(np.float64).reshape(-1, 3, cfg.dim)
    mod[1, 2, :] = 0.0
    mod[2, 2, :] = 0.0                          # only the self-attention gate is on
    o = FlashMap(cfg, w, mod.reshape(-1), True)
    st = o.new_state()
    o.context_append(st, S.gen_features(S.streams(13)["features"], 2, cfg.feat_dim), 0)
    r = o.draft(st, 1, 2)
    m = mod[0]
    hn = (o.h0 - o.h0.mean()) / np.sqrt(o.h0.var() + cfg.ln_eps) * (1 + m[0]) + m[1]
    v = C.bf16_to_f64(w["layers.0.self_attn.v_proj.weight"]) @ hn
    want = o.h0 + m[2] * (C.bf16_to_f64(w["layers.0.self_attn.o_proj.weight"]) @ v)
    np.testing.assert_allclose(r.hidden[0], np.tile(want, (cfg.block, 1)), rtol=1e-13)


def test_flashmap_single_key_cross_attention_is_anchor_v():
    """At pos = 0 the cross keys are the anchor slot alone: the output is its
    (f16-stored) value row."""
    cfg = micro_flashmap(n_layers=1)
    w = raw_weights(cfg, 14)
    mod = S.gen_modulation(cfg, 14).astype(np.float64).reshape(-1, 3, cfg.dim)
    mod[0, 2, :] = 0.0
    mod[2, 2, :] = 0.0                          # only the cross-attention gate is on
    o = FlashMap(cfg, w, mod.reshape(-1), True)
    st = o.new_state()
    r = o.draft(st, 9, 0)
    E = C.q8_0_dequant(w["token_embd.weight"], cfg.target_dim)
    a = C.bf16_to_f64(w["anchor_proj.weight"]) @ E[9] + C.bf16_to_f64(w["anchor_proj.bias"])
    a = a / np.sqrt(np.mean(a * a) + cfg.rms_eps) * C.bf16_to_f64(w["anchor_norm.weight"])
    v = (C.bf16_to_f64(w["layers.0.cross_attn.v_proj.weight"]) @ a).astype(np.float16).astype(np.float64)
    want = o.h0 + mod[1, 2] * (C.bf16_to_f64(w["layers.0.cross_attn.o_proj.weight"]) @ v)
    np.testing.assert_allclose(r.hidden[0], np.tile(want, (cfg.block, 1)), rtol=1e-13)


def test_flashmap_append_chunking_and_rewind():
    cfg = micro_flashmap()
    w = raw_weights(cfg, 15)
    o = FlashMap(cfg, w, S.gen_modulation(cfg, 15), True)
    feats = S.gen_features(S.streams(15)["features"], 7, cfg.feat_dim)
    a = o.new_state()
    o.context_append(a, feats, 0)
    b = o.new_state()
    o.context_append(b, feats[:1], 0)
    o.context_append(b, feats[1:], 1)
    c = o.new_state()
    o.context_append(c, feats[:5], 0)
    o.context_append(c, S.gen_features(S.streams(99)["features"], 2, cfg.feat_dim), 5)
    o.context_append(c, feats[3:], 3)            # rewind to 3, re-append the same rows
    for l in range(cfg.n_layers):
        for s in (b, c):
            np.testing.assert_array_equal(a.k[l][:7], s.k[l][:7])
            np.testing.assert_array_equal(a.v[l][:7], s.v[l][:7])
    assert a.length == b.length == c.length == 7
    with pytest.raises(ValueError):
        o.context_append(a, S.gen_features(S.streams(1)["features"], cfg.max_ctx - 7 - cfg.block, cfg.feat_dim), 7)


def test_dflash_matches_brute_force():
    cfg = micro_dflash()
    w = raw_weights(cfg, 21)
    feats = S.gen_features(S.streams(21)["features"], 4, cfg.feat_dim)
    o = DFlash(cfg, w)
    b = brute.BruteDFlash(cfg, w)
    st = o.new_state()
    o.context_append(st, feats, 0)
    b.append(feats, 0)
    for pos, anchor in ((4, 5), (0, 2)):
        if pos == 0:
            st = o.new_state()
            b = brute.BruteDFlash(cfg, w)
        r = o.draft(st, anchor, pos)
        toks, logits, Y, hidden = b.draft(anchor, pos)
        for l in range(cfg.n_layers):
            np.testing.assert_allclose(r.hidden[l], hidden[l], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(r.head_out, Y, rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(r.logits, logits, rtol=1e-10, atol=1e-13)
        assert r.tokens.tolist() == toks


def test_dflash_cached_context_equals_reprojected_context():
    """The page's two routes: retained per-layer context K/V (context.attend)
    and re-projecting H_ctx inside every layer give the same block."""
    cfg = micro_dflash()
    w = raw_weights(cfg, 22)
    feats = S.gen_features(S.streams(22)["features"], 6, cfg.feat_dim)
    o = DFlash(cfg, w)
    st = o.new_state()
    o.context_append(st, feats[:2], 0)
    o.context_append(st, feats[2:], 2)
    r = o.draft(st, 4, 6)
    hc = o.build_context(feats)
    Hd = o.build_block(4)
    for i in range(cfg.n_layers):
        nc = C.rms_norm(hc, o.w[f"bb.{i}.attn_norm"], cfg.rms_eps)
        Hd = o.layer(i, Hd, nc @ o.w[f"bb.{i}.k"], nc @ o.w[f"bb.{i}.v"])
        np.testing.assert_allclose(r.hidden[i], Hd, rtol=1e-12)
