"""Pins of the time-conditioning oracle (flashmap_drafter.js,
``timeConditioning``) against closed forms, an independent library routine and
a brute-force restatement on micro dims.  CPU only."""
from __future__ import annotations

import math

import numpy as np
import scipy.special

import brute
import fm_synth as S
from oracle import timecond as TC


def micro_cfg():
    return S.DrafterConfig(S.VARIANT_FLASHMAP, dim=8, n_heads=2, head_dim=4, n_layers=2, ff_dim=12, block=4,
                           target_dim=32, n_taps=2, vocab=16, lm_format=S.LM_BF16, max_ctx=24)


def raw(w):
    return {n: t.data for n, t in w.items()}


def test_sinusoid_at_time_zero_is_ones_then_zeros():
    e = TC.sinusoidal_embedding(0.0, 16, 1000.0)
    np.testing.assert_array_equal(e, np.r_[np.ones(8), np.zeros(8)])


def test_sinusoid_worked_values():
    # time 1, width 4, scale 1: half 2, frequencies 1 and exp(-ln(10000) / 2) = 1 / 100
    e = TC.sinusoidal_embedding(1.0, 4, 1.0)
    np.testing.assert_allclose(e, [0.5403023058681398, 0.9999500004166653, 0.8414709848078965,
                                   0.009999833334166664], rtol=0, atol=1e-15)


def test_silu_matches_library_logistic():
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(TC.silu(x), x * scipy.special.expit(x), rtol=1e-14, atol=1e-300)
    assert TC.silu(np.array([0.0]))[0] == 0.0


def test_matches_brute_force_on_micro_dims():
    cfg = micro_cfg()
    w = raw(S.gen_time_cond_weights(cfg, 5, time_dim=6, cond_dim=5, std=0.3))
    got = TC.time_conditioning(w, cfg.n_layers, cfg.dim, 6, 1000.0, 0.0, 1.0)
    want = brute.time_conditioning(w, cfg.n_layers, 6, 1000.0, 0.0, 1.0)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
    # an intermediate jump (s, t not 0 / 1) agrees as well
    got = TC.time_conditioning(w, cfg.n_layers, cfg.dim, 6, 1000.0, 0.25, 0.75)
    want = brute.time_conditioning(w, cfg.n_layers, 6, 1000.0, 0.25, 0.75)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_zero_adaln_weights_give_the_biases_in_table_order():
    cfg = micro_cfg()
    w = raw(S.gen_time_cond_weights(cfg, 6, time_dim=6, cond_dim=5, std=0.3))
    names = TC.adaln_names(cfg.n_layers)
    assert names[:3] == ["layers.0.self_attn_adaln.linear", "layers.0.cross_attn_adaln.linear",
                         "layers.0.mlp_adaln.linear"] and names[-1] == "final_adaln.linear"
    biases = []
    for i, n in enumerate(names):
        w[n + ".weight"] = np.zeros_like(w[n + ".weight"])
        bits = S.f32_to_bf16_bits(np.arange(3 * cfg.dim, dtype=np.float32) + 100 * i)
        w[n + ".bias"] = bits
        biases.append(S.bf16_bits_to_f32(bits))             # the values the bf16 patterns hold
    got = TC.time_conditioning(w, cfg.n_layers, cfg.dim, 6, 1000.0, 0.0, 1.0)
    np.testing.assert_array_equal(got, np.concatenate(biases).astype(np.float64))


def test_constant_embeddings_make_the_table_independent_of_the_jump():
    cfg = micro_cfg()
    w = raw(S.gen_time_cond_weights(cfg, 7, time_dim=6, cond_dim=5, std=0.3))
    for p in ("time_embed", "jump_embed"):
        w[p + ".linear_2.weight"] = np.zeros_like(w[p + ".linear_2.weight"])
    a = TC.time_conditioning(w, cfg.n_layers, cfg.dim, 6, 1000.0, 0.0, 1.0)
    b = TC.time_conditioning(w, cfg.n_layers, cfg.dim, 6, 1000.0, 0.3, 0.9)
    np.testing.assert_array_equal(a, b)
    # and cond is SiLU of the two linear_2 biases: check the first block by hand
    bt = S.bf16_bits_to_f32(w["time_embed.linear_2.bias"]).astype(np.float64)
    bj = S.bf16_bits_to_f32(w["jump_embed.linear_2.bias"]).astype(np.float64)
    cond = [(x + y) / (1 + math.exp(-(x + y))) for x, y in zip(bt, bj)]
    W = S.bf16_bits_to_f32(w["layers.0.self_attn_adaln.linear.weight"]).astype(np.float64)
    B = S.bf16_bits_to_f32(w["layers.0.self_attn_adaln.linear.bias"]).astype(np.float64)
    first = [sum(W[m, k] * cond[k] for k in range(len(cond))) + B[m] for m in range(3 * cfg.dim)]
    np.testing.assert_allclose(a[:3 * cfg.dim], first, rtol=1e-12, atol=1e-14)
