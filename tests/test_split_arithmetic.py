"""The number formats the CUDA path rests on, checked on the host with numpy's
IEEE half / bfloat16-by-bits arithmetic (no GPU):

* the Q8_0 lm_head forms each weight q * d (int8 times the f16 block scale) as
  hi = rn16(q * d) and lo = rn16(q * d - hi) -- one f16 multiply and one fused
  multiply-add -- and feeds hi and lo to the tensor cores as two A operands;
  hi + lo must equal q * d exactly wherever lo is a normal f16, and be within
  half a subnormal step otherwise;
* the activations are split the same way into bf16 (GEMV) or f16 (lm_head)
  hi + lo; the pair must carry about 16 (bf16) / 22 (f16) bits of the f32 value
  (f16: down to an absolute floor of 2^-25, where the residual is subnormal).

These are the arithmetic facts the kernels' hi / lo operands rely on (the GPU
parity tests check the kernels themselves against the oracle); the first check
would fail for a split that rounds the residual twice or drops it."""
from __future__ import annotations

import numpy as np


def rn16(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float16)


def q8_split(q: np.ndarray, d: np.ndarray):
    # q * d is exact in f32 (8 + 11 significant bits); the residual q * d - hi is
    # exact in f32 as well, so one rounding to f16 models the fused multiply-add
    prod = q.astype(np.float32) * d.astype(np.float32)
    hi = rn16(prod)
    lo = rn16(prod - hi.astype(np.float32))
    return prod, hi, lo


def test_q8_product_split_is_exact():
    rng = np.random.default_rng(7)
    q = np.arange(-128, 128, dtype=np.int32)[None, :]
    # block scales spanning the range a Q8_0 table uses (max |w| / 127 for |w| up to ~8)
    d = rng.uniform(2.0 ** -12, 2.0 ** -4, size=(4096, 1)).astype(np.float16)
    prod, hi, lo = q8_split(np.broadcast_to(q, (4096, 256)), np.broadcast_to(d, (4096, 256)))
    total = hi.astype(np.float64) + lo.astype(np.float64)
    exact = prod.astype(np.float64)
    normal_lo = (np.abs(lo.astype(np.float64)) >= 2.0 ** -14) | (lo == 0)
    assert np.array_equal(total[normal_lo], exact[normal_lo])
    # a subnormal residual loses at most half a subnormal step (2^-25)
    assert np.max(np.abs(total - exact)) <= 2.0 ** -25
    # and the split is needed: hi alone is off by up to half an f16 ulp of the product
    assert np.max(np.abs(hi.astype(np.float64) - exact) / np.maximum(np.abs(exact), 1e-30)) > 2.0 ** -13


def bf16_rn(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) & np.uint32(0xFFFF0000)).view(np.float32)


def test_activation_splits_carry_f32_precision():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-6, 6, 200000))).astype(np.float32)
    hi = bf16_rn(x)
    lo = bf16_rn(x - hi)
    rel = np.abs((hi.astype(np.float64) + lo.astype(np.float64)) - x) / np.abs(x)
    assert rel.max() < 2.0 ** -16          # bf16 hi + lo: ~17 bits
    y = x[np.abs(x) < 6e4]                  # inside f16's range
    h16 = rn16(y)
    l16 = rn16(y - h16.astype(np.float32))
    err16 = np.abs((h16.astype(np.float64) + l16.astype(np.float64)) - y)
    # f16 hi + lo: ~22 bits, down to the absolute floor of a subnormal residual (half of 2^-24)
    assert np.all(err16 <= np.maximum(2.0 ** -21 * np.abs(y), 2.0 ** -25))
