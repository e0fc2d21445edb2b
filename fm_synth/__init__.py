"""Seeded synthetic inputs for the block-parallel drafter (FlashMap / DFlash kind).

This module is the ONE place both sides of the parity check draw from: the
CUDA path (bench, GPU tests) and the CPU oracle (tests) get their weights,
modulation table, feature rows, anchors and target tokens from here.  It holds
none of the drafter's arithmetic: it only draws random numbers, rounds them to
the storage formats the drafter consumes (bf16, GGUF Q8_0 blocks) and packs
bytes.  Nothing here normalises, projects, rotates or attends.

Workload shapes follow the source pages:
  * flashmap_drafter.js (diskformer 0.6.6), ``CFG`` and the tapped-layer list:
    dim 2048, 16 x 128 heads, 6 layers, ff 8192, block 16, target dim 2560,
    5 taps, RoPE base 1e4, eps 1e-6 / 1e-6 / 1e-5.
  * module-dflash.ts (mlx-bun 1.0.0), ``DEFAULT_DFLASH_CONFIG`` and
    ``initFromDims``: gamma 5, d 1024, 5 layers, 8 heads, ffMult 2, 4 taps,
    weights stored [in, out].
  * Q8_0 block: f16 scale then 32 int8 (34 bytes), as the MTP head's loader
    reads GGUF type 8 (ternary_bonsai_2_mtp.js, ``loadWeights``).

Distributions (the workload recipe): weights and biases bf16(N(0, 0.02)); norm
weights bf16(1 + N(0, 0.02)); adaLN modulation f32 N(0, 0.1); feature rows
f32 N(0, 1); anchors uniform in [0, V); the tied token table is bf16(N(0, 0.02))
or its Q8_0 quantisation.  Every role draws from its own PCG64 stream spawned
from ``SeedSequence(seed)`` so a role can be regenerated without the others.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np

# dtype tags shared with the C-ABI (include/fm.h: FM_DTYPE_*)
DT_BF16 = 0
DT_Q8_0 = 1
DT_F32 = 2

VARIANT_FLASHMAP = 0
VARIANT_DFLASH = 1
LM_BF16 = 0
LM_Q8_0 = 1


@dataclasses.dataclass(frozen=True)
class DrafterConfig:
    variant: int
    dim: int
    n_heads: int
    head_dim: int
    n_layers: int
    ff_dim: int
    block: int
    target_dim: int
    n_taps: int
    vocab: int
    lm_format: int
    max_ctx: int
    max_seqs: int = 1
    rope_theta: float = 10000.0
    ln_eps: float = 1e-6
    rms_eps: float = 1e-6
    qk_eps: float = 1e-5

    @property
    def feat_dim(self) -> int:
        return self.n_taps * self.target_dim

    def replace(self, **kw) -> "DrafterConfig":
        return dataclasses.replace(self, **kw)


# --- named workloads -------------------------------------------------------

def tiny_config(max_ctx: int = 128) -> DrafterConfig:
    """Tiny FlashMap-shaped drafter: D 256, 4 x 64 heads, 2 layers, ff 1024,
    block 16, target dim 320, 3 taps (960), vocab 4096 bf16 table."""
    return DrafterConfig(VARIANT_FLASHMAP, 256, 4, 64, 2, 1024, 16, 320, 3, 4096, LM_BF16, max_ctx)


def flashmap_4b_config(max_ctx: int = 1024 + 17 + 34, max_seqs: int = 1) -> DrafterConfig:
    """FlashMap-Qwen3-4B shape (flashmap_drafter.js ``CFG``), Q8_0 vocab 151936."""
    return DrafterConfig(VARIANT_FLASHMAP, 2048, 16, 128, 6, 8192, 16, 2560, 5, 151936, LM_Q8_0,
                         max_ctx, max_seqs)


def dflash_config(max_ctx: int = 4096 + 6 * 200 + 16) -> DrafterConfig:
    """DFlash KV-injection drafter (module-dflash.ts defaults): d 1024, 8 heads
    x 128, 5 layers, ff 2 x 1024, gamma 5, 4 taps of 2560, bf16 vocab 262144."""
    return DrafterConfig(VARIANT_DFLASH, 1024, 8, 128, 5, 2048, 5, 2560, 4, 262144, LM_BF16, max_ctx,
                         rms_eps=1e-6)


# --- storage-format rounding (data preparation, not drafter arithmetic) ----

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round f32 values to bf16 (nearest, ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """GGUF Q8_0 blocks of a [rows, cols] f32 matrix: per 32 values an f16
    scale d = max|x| / 127 and int8 q = round(x / d).  Returns uint8
    [rows, cols / 32 * 34] (little-endian f16 d, then 32 int8)."""
    rows, cols = x.shape
    assert cols % 32 == 0
    nb = cols // 32
    blk = x.reshape(rows, nb, 32).astype(np.float32)
    amax = np.abs(blk).max(axis=2)
    d = (amax / 127.0).astype(np.float16)
    d32 = d.astype(np.float32)
    inv = np.divide(1.0, d32, out=np.zeros_like(d32), where=d32 != 0)
    q = np.clip(np.rint(blk * inv[:, :, None]), -127, 127).astype(np.int8)
    out = np.empty((rows, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = d.reshape(rows, nb, 1).view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:34] = q.view(np.uint8)
    return out.reshape(rows, nb * 34)


# --- streams ---------------------------------------------------------------

_ROLES = ("weights", "modulation", "features", "tokens", "workload")


def streams(seed: int) -> Dict[str, np.random.Generator]:
    kids = np.random.SeedSequence(seed).spawn(len(_ROLES))
    return {r: np.random.Generator(np.random.PCG64(s)) for r, s in zip(_ROLES, kids)}


def _normal(rng: np.random.Generator, shape, std: float, mean: float = 0.0) -> np.ndarray:
    n = int(np.prod(shape))
    v = rng.standard_normal(n, dtype=np.float32)
    v *= np.float32(std)
    if mean:
        v += np.float32(mean)
    return v.reshape(shape)


# --- tensor lists ----------------------------------------------------------

def flashmap_tensor_specs(cfg: DrafterConfig) -> List[Tuple[str, Tuple[int, ...], str]]:
    """(name, shape, kind) in generation order.  Names follow the drafter's
    checkpoint (flashmap_drafter.js ``init``/``extendContext``); weights are
    [out][in].  kind: w = N(0, .02), b = bias N(0, .02), n = 1 + N(0, .02),
    t = the tied token table."""
    D, hd, F, Ht, m = cfg.dim, cfg.head_dim, cfg.ff_dim, cfg.target_dim, cfg.n_taps
    s: List[Tuple[str, Tuple[int, ...], str]] = [
        ("fc.weight", (D, m * Ht), "w"),
        ("hidden_norm.weight", (D,), "n"),
        ("anchor_proj.weight", (D, Ht), "w"),
        ("anchor_proj.bias", (D,), "b"),
        ("anchor_norm.weight", (D,), "n"),
        ("state_norm.weight", (Ht,), "n"),
        ("x_embed.weight", (D, Ht), "w"),
        ("x_embed.bias", (D,), "b"),
    ]
    for l in range(cfg.n_layers):
        p = f"layers.{l}."
        for att in ("self_attn", "cross_attn"):
            for x in ("q", "k", "v", "o"):
                s.append((f"{p}{att}.{x}_proj.weight", (D, D), "w"))
            s.append((f"{p}{att}.q_norm.weight", (hd,), "n"))
            s.append((f"{p}{att}.k_norm.weight", (hd,), "n"))
        s += [(f"{p}mlp.fc1.weight", (F, D), "w"), (f"{p}mlp.fc1.bias", (F,), "b"),
              (f"{p}mlp.fc2.weight", (D, F), "w"), (f"{p}mlp.fc2.bias", (D,), "b")]
    s += [("head.weight", (Ht, D), "w"), ("head.bias", (Ht,), "b"),
          ("token_embd.weight", (cfg.vocab, Ht), "t")]
    return s


def dflash_tensor_specs(cfg: DrafterConfig) -> List[Tuple[str, Tuple[int, ...], str]]:
    """(name, shape, kind) in the checkpoint's name order (module-dflash.ts
    ``buildNames``), [in, out] layout as ``initFromDims`` makes them.  The
    sequential-head (markov / rnn) and confidence tensors are not part of the
    parallel draft pass and are not generated."""
    d, F, H, m, g = cfg.dim, cfg.ff_dim, cfg.target_dim, cfg.n_taps, cfg.block
    s: List[Tuple[str, Tuple[int, ...], str]] = []
    for i in range(cfg.n_layers):
        p = f"bb.{i}."
        s += [(p + "attn_norm", (d,), "n"), (p + "q", (d, d), "w"), (p + "k", (d, d), "w"),
              (p + "v", (d, d), "w"), (p + "o", (d, d), "w"), (p + "ff_norm", (d,), "n"),
              (p + "gate", (d, F), "w"), (p + "up", (d, F), "w"), (p + "down", (F, d), "w")]
    s += [("W_c", (m * H, d), "w"), ("ctx_norm", (d,), "n"), ("tok_proj", (H, d), "w"),
          ("mask_emb", (g - 1, d), "w"), ("block_pos", (g, d), "w"), ("out_norm", (d,), "n"),
          ("out_proj", (d, H), "w"), ("token_embd.weight", (cfg.vocab, H), "t")]
    return s


def tensor_specs(cfg: DrafterConfig):
    return flashmap_tensor_specs(cfg) if cfg.variant == VARIANT_FLASHMAP else dflash_tensor_specs(cfg)


@dataclasses.dataclass
class Tensor:
    name: str
    shape: Tuple[int, ...]   # logical shape (for Q8_0: [rows, cols] of values)
    dtype: int               # DT_BF16 / DT_Q8_0 / DT_F32
    data: np.ndarray         # uint16 bf16 bits, uint8 Q8_0 bytes, or f32


def _gen_table(rng, cfg: DrafterConfig) -> Tensor:
    V, H = cfg.vocab, cfg.target_dim
    if cfg.lm_format == LM_BF16:
        bits = np.empty((V, H), dtype=np.uint16)
        step = 16384
        for r0 in range(0, V, step):
            r1 = min(V, r0 + step)
            bits[r0:r1] = f32_to_bf16_bits(_normal(rng, (r1 - r0, H), 0.02))
        return Tensor("token_embd.weight", (V, H), DT_BF16, bits)
    raw = np.empty((V, H // 32 * 34), dtype=np.uint8)
    step = 8192
    for r0 in range(0, V, step):
        r1 = min(V, r0 + step)
        x = bf16_bits_to_f32(f32_to_bf16_bits(_normal(rng, (r1 - r0, H), 0.02)))
        raw[r0:r1] = quantize_q8_0(x)
    return Tensor("token_embd.weight", (V, H), DT_Q8_0, raw)


def gen_weights(cfg: DrafterConfig, seed: int) -> Dict[str, Tensor]:
    rng = streams(seed)["weights"]
    out: Dict[str, Tensor] = {}
    for name, shape, kind in tensor_specs(cfg):
        if kind == "t":
            out[name] = _gen_table(rng, cfg)
        elif kind == "n":
            out[name] = Tensor(name, shape, DT_BF16, f32_to_bf16_bits(_normal(rng, shape, 0.02, 1.0)))
        else:
            out[name] = Tensor(name, shape, DT_BF16, f32_to_bf16_bits(_normal(rng, shape, 0.02)))
    return out


def gen_modulation(cfg: DrafterConfig, seed: int) -> np.ndarray:
    """adaLN table [(3L + 1) * 3 * D] f32, blocks [scale D | shift D | gate D]."""
    rng = streams(seed)["modulation"]
    return _normal(rng, ((3 * cfg.n_layers + 1) * 3 * cfg.dim,), 0.1)


def gen_features(rng: np.random.Generator, n: int, width: int) -> np.ndarray:
    return _normal(rng, (n, width), 1.0)


def gen_anchor(rng: np.random.Generator, vocab: int) -> int:
    return int(rng.integers(0, vocab))


def targets_with_flip(drafts: np.ndarray, k: int, flip: int, vocab: int,
                      rng: np.random.Generator) -> np.ndarray:
    """Target tokens [k + 1] that agree with ``drafts`` on slots < flip and
    differ at slot ``flip`` (if flip < k); slot k (the bonus row) is random.
    The longest matching prefix is then exactly ``flip``."""
    t = np.array(drafts[:k], dtype=np.int64).copy()
    t = np.concatenate([t, [int(rng.integers(0, vocab))]])
    if flip < k:
        t[flip] = (int(drafts[flip]) + 1 + int(rng.integers(0, vocab - 1))) % vocab
        for j in range(flip + 1, k):
            t[j] = int(rng.integers(0, vocab))
    return t.astype(np.int32)


def batched_lengths(rng: np.random.Generator, n_seqs: int = 32, lo: int = 512, hi: int = 8192):
    """Per-sequence context lengths, uniform in [lo, hi]."""
    return rng.integers(lo, hi + 1, size=n_seqs).astype(np.int64)


# ---------------------------------------------------------------- time conditioning

def time_cond_specs(cfg: DrafterConfig, time_dim: int = 256, cond_dim: int = 256):
    """(name, shape) of the FlashMap time-conditioning linears: the sinusoid's
    two MLPs (time_embed for s, jump_embed for t) and one adaLN linear per
    norm, in table order."""
    s = []
    for p in ("time_embed", "jump_embed"):
        s += [(f"{p}.linear_1.weight", (cond_dim, time_dim)), (f"{p}.linear_1.bias", (cond_dim,)),
              (f"{p}.linear_2.weight", (cond_dim, cond_dim)), (f"{p}.linear_2.bias", (cond_dim,))]
    names = [f"layers.{l}.{n}.linear" for l in range(cfg.n_layers)
             for n in ("self_attn_adaln", "cross_attn_adaln", "mlp_adaln")] + ["final_adaln.linear"]
    for n in names:
        s += [(n + ".weight", (3 * cfg.dim, cond_dim)), (n + ".bias", (3 * cfg.dim,))]
    return s


def gen_time_cond_weights(cfg: DrafterConfig, seed: int, time_dim: int = 256, cond_dim: int = 256,
                          std: float = 0.02) -> Dict[str, Tensor]:
    """bf16(N(0, std)) time-conditioning weights and biases (seeded stream of their own)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    return {n: Tensor(n, shape, DT_BF16, f32_to_bf16_bits(_normal(rng, shape, std)))
            for n, shape in time_cond_specs(cfg, time_dim, cond_dim)}


# ---------------------------------------------------------------- DFlash sequential head

def gen_seq_head_weights(cfg: DrafterConfig, seed: int, variant: str = "markov", rank: int = 256,
                         w1_std: float = 1.0, w2_std: float = 0.05) -> Dict[str, Tensor]:
    """The sequential logit head (markov.w1 [V, r], markov.w2 [r, V]; with
    variant "rnn" also rnn.wH [r, r], rnn.bH [r], rnn.wO [r, V]) and the
    confidence head (conf.w [d + r, 1], conf.b [1]), bf16.  The bias e1 . w2
    is scaled to the size of the base logits so that it moves some argmaxes."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 11])))
    V, d = cfg.vocab, cfg.dim
    spec = [("markov.w1", (V, rank), w1_std), ("markov.w2", (rank, V), w2_std),
            ("conf.w", (d + rank, 1), 0.02), ("conf.b", (1,), 0.1)]
    if variant == "rnn":
        spec += [("rnn.wH", (rank, rank), 0.05), ("rnn.bH", (rank,), 0.05), ("rnn.wO", (rank, V), 0.1)]
    out = {}
    for n, shape, std in spec:
        out[n] = Tensor(n, shape, DT_BF16, f32_to_bf16_bits(_normal(rng, shape, std)))
    return out


# --- the MTP draft head (ternary_bonsai_2_mtp.js, ``MCFG`` / ``MTP_HEAD``) --

@dataclasses.dataclass(frozen=True)
class MtpConfig:
    hidden: int = 5120
    inter: int = 17408
    n_heads: int = 24
    n_kv_heads: int = 4
    head_dim: int = 256
    rot_dims: int = 64
    theta: float = 1e7
    eps: float = 1e-6
    vocab: int = 248320
    kv_cap: int = 4096 + 64
    max_rows: int = 8

    def replace(self, **kw) -> "MtpConfig":
        return dataclasses.replace(self, **kw)


def mtp_config(kv_cap: int = 4096 + 64) -> MtpConfig:
    """The page's MTP head: H 5120, I 17408, 24 q heads and 4 KV heads of 256,
    NEOX RoPE on 64 dims with theta 1e7, eps 1e-6, vocab 248320, M <= 8 rows."""
    return MtpConfig(kv_cap=kv_cap)


def mtp_micro_config(kv_cap: int = 96) -> MtpConfig:
    """A small MTP head of the same structure (the oracle runs it in seconds)."""
    return MtpConfig(hidden=256, inter=512, n_heads=4, n_kv_heads=2, head_dim=64, rot_dims=32, theta=1e4,
                     vocab=4096, kv_cap=kv_cap)


def mtp_tensor_specs(cfg: MtpConfig) -> List[Tuple[str, Tuple[int, ...], str]]:
    """(name, [N, K] or [n], kind): "q" a Q8_0 matrix (y = W x, W [N][K]), "n" an
    f32 norm weight, "e" the bf16 embedding table, "l" the Q8_0 lm_head."""
    H, I, nh, nkv, hd = cfg.hidden, cfg.inter, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    return [("eh_proj", (H, 2 * H), "q"), ("attn_q", (nh * 2 * hd, H), "q"), ("attn_k", (nkv * hd, H), "q"),
            ("attn_v", (nkv * hd, H), "q"), ("attn_output", (H, nh * hd), "q"), ("ffn_gate", (I, H), "q"),
            ("ffn_up", (I, H), "q"), ("ffn_down", (H, I), "q"),
            ("enorm", (H,), "n"), ("hnorm", (H,), "n"), ("attn_norm", (H,), "n"), ("attn_q_norm", (hd,), "n"),
            ("attn_k_norm", (hd,), "n"), ("post_attention_norm", (H,), "n"), ("shared_head_norm", (H,), "n"),
            ("token_embd", (cfg.vocab, H), "e"), ("lm_head", (cfg.vocab, H), "l")]


def gen_mtp_weights(cfg: MtpConfig, seed: int) -> Dict[str, Tensor]:
    """Matrices N(0, 0.02) quantised to Q8_0, norms f32 1 + N(0, 0.02), the
    embedding table bf16(N(0, 1)) (embedding rows of unit scale, as a trunk's
    are), the lm_head N(0, 0.02) quantised to Q8_0.  Large tensors are drawn
    and quantised in row blocks."""
    rng = streams(seed)["weights"]
    out: Dict[str, Tensor] = {}
    for name, shape, kind in mtp_tensor_specs(cfg):
        if kind == "n":
            out[name] = Tensor(name, shape, DT_F32, _normal(rng, shape, 0.02, 1.0))
        elif kind == "e":
            bits = np.empty(shape, dtype=np.uint16)
            for r0 in range(0, shape[0], 16384):
                r1 = min(shape[0], r0 + 16384)
                bits[r0:r1] = f32_to_bf16_bits(_normal(rng, (r1 - r0, shape[1]), 1.0))
            out[name] = Tensor(name, shape, DT_BF16, bits)
        else:
            rows, cols = shape
            raw = np.empty((rows, cols // 32 * 34), dtype=np.uint8)
            for r0 in range(0, rows, 4096):
                r1 = min(rows, r0 + 4096)
                raw[r0:r1] = quantize_q8_0(_normal(rng, (r1 - r0, cols), 0.02))
            out[name] = Tensor(name, shape, DT_Q8_0, raw)
    return out


def gen_mtp_hidden(rng: np.random.Generator, n: int, hidden: int) -> np.ndarray:
    """Rows standing in for the trunk's output-normed hidden states: f32 N(0, 1)."""
    return rng.standard_normal((n, hidden), dtype=np.float32)
