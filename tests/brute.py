"""Brute-force scalar restatement of the drafter on micro dims, used to pin the
numpy oracle.  Pure Python: explicit index loops, ``struct`` for the storage
formats and ``math`` for the transcendental functions.  It imports nothing from
oracle/ or from the CUDA package, so a dropped term, a wrong sign, a swapped
index or a transposed operand in the oracle disagrees with it.

Sources: flashmap_drafter.js (diskformer 0.6.6): ``extendContext``, ``draft``
and the WGSL kernels it dispatches; module-dflash.ts (mlx-bun 1.0.0): Eq 2,
Eq 3, ``#buildBlock``, ``#layer``.
"""
from __future__ import annotations

import math
import struct


def bf(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def half(x: float) -> float:
    return struct.unpack("<e", struct.pack("<e", x))[0]


def mat(bits2d):
    return [[bf(b) for b in row] for row in bits2d]


def vec(bits1d):
    return [bf(b) for b in bits1d]


def q8_row(raw_row, ncols: int):
    out = []
    raw = bytes(int(b) for b in raw_row)
    for blk in range(ncols // 32):
        o = blk * 34
        d = struct.unpack("<e", raw[o:o + 2])[0]
        qs = struct.unpack("32b", raw[o + 2:o + 34])
        out.extend(d * q for q in qs)
    return out


def matvec(W, x, b=None):
    """W is [out][in]: y[m] = sum_k W[m][k] x[k] (+ b[m])."""
    y = []
    for m in range(len(W)):
        s = 0.0
        row = W[m]
        for k in range(len(x)):
            s += row[k] * x[k]
        y.append(s + (b[m] if b is not None else 0.0))
    return y


def vecmat(x, W):
    """W is [in][out]: y[n] = sum_k x[k] W[k][n]."""
    n_out = len(W[0])
    y = [0.0] * n_out
    for k in range(len(x)):
        for n in range(n_out):
            y[n] += x[k] * W[k][n]
    return y


def rmsn(x, w, eps):
    ms = 0.0
    for v in x:
        ms += v * v
    r = 1.0 / math.sqrt(ms / len(x) + eps)
    return [x[i] * r * w[i] for i in range(len(x))]


def lnmod(x, scale, shift, eps):
    n = len(x)
    mu = sum(x) / n
    var = 0.0
    for v in x:
        var += (v - mu) * (v - mu)
    r = 1.0 / math.sqrt(var / n + eps)
    return [(x[i] - mu) * r * (1.0 + scale[i]) + shift[i] for i in range(n)]


def headnorm_rope(x, w, eps, hd, pos, theta, rope=True):
    out = list(x)
    for h in range(len(x) // hd):
        seg = x[h * hd:(h + 1) * hd]
        ms = 0.0
        for v in seg:
            ms += v * v
        r = 1.0 / math.sqrt(ms / hd + eps)
        y = [seg[i] * w[i] * r for i in range(hd)]
        if rope:
            for i in range(hd // 2):
                ang = pos * theta ** (-2.0 * i / hd)
                c, s = math.cos(ang), math.sin(ang)
                a0, a1 = y[2 * i], y[2 * i + 1]
                y[2 * i] = a0 * c - a1 * s
                y[2 * i + 1] = a1 * c + a0 * s
        out[h * hd:(h + 1) * hd] = y
    return out


def attend(qs, ks, vs, hd):
    """qs: list of query rows, ks/vs: lists of key/value rows; unmasked."""
    nh = len(qs[0]) // hd
    outs = []
    for q in qs:
        o = [0.0] * len(q)
        for h in range(nh):
            sc = []
            for kr in ks:
                s = 0.0
                for d in range(hd):
                    s += q[h * hd + d] * kr[h * hd + d]
                sc.append(s / math.sqrt(hd))
            mx = max(sc)
            es = [math.exp(s - mx) for s in sc]
            tot = sum(es)
            for d in range(hd):
                acc = 0.0
                for j, vr in enumerate(vs):
                    acc += es[j] * vr[h * hd + d]
                o[h * hd + d] = acc / tot
        outs.append(o)
    return outs


def gelu(x):
    return 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))


def gelu_tanh(x):
    return 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x * x * x)))


def argmax(row):
    best, bi = row[0], 0
    for i in range(1, len(row)):
        if row[i] > best:
            best, bi = row[i], i
    return bi


class BruteFlashMap:
    def __init__(self, cfg, w, modulation, table_q8):
        self.c = cfg
        self.W = {}
        for n, a in w.items():
            if n == "token_embd.weight":
                continue
            self.W[n] = mat(a) if a.ndim == 2 else vec(a)
        raw = w["token_embd.weight"]
        self.E = [q8_row(r, cfg.target_dim) for r in raw] if table_q8 else mat(raw)
        D = cfg.dim
        self.mod = [float(v) for v in modulation]
        u = [0.0] * cfg.target_dim
        for row in self.E:
            for i, v in enumerate(row):
                u[i] += v
        u = [v / len(self.E) for v in u]
        s = rmsn(u, self.W["state_norm.weight"], cfg.rms_eps)
        self.h0 = matvec(self.W["x_embed.weight"], s, self.W["x_embed.bias"])
        self.K = [dict() for _ in range(cfg.n_layers)]
        self.V = [dict() for _ in range(cfg.n_layers)]
        self.D = D

    def modpart(self, n, part):
        D = self.D
        return self.mod[(3 * n + part) * D:(3 * n + part + 1) * D]

    def _kv(self, l, x, p):
        c = self.c
        pre = f"layers.{l}.cross_attn."
        k = matvec(self.W[pre + "k_proj.weight"], x)
        v = matvec(self.W[pre + "v_proj.weight"], x)
        k = headnorm_rope(k, self.W[pre + "k_norm.weight"], c.qk_eps, c.head_dim, p, c.rope_theta)
        self.K[l][p] = [half(a) for a in k]
        self.V[l][p] = [half(a) for a in v]

    def append(self, feats, start):
        c = self.c
        for t, f in enumerate(feats):
            x = matvec(self.W["fc.weight"], [float(a) for a in f])
            x = rmsn(x, self.W["hidden_norm.weight"], c.rms_eps)
            for l in range(c.n_layers):
                self._kv(l, x, start + t)

    def draft(self, anchor, pos):
        c = self.c
        hd = c.head_dim
        a = matvec(self.W["anchor_proj.weight"], self.E[anchor], self.W["anchor_proj.bias"])
        a = rmsn(a, self.W["anchor_norm.weight"], c.rms_eps)
        for l in range(c.n_layers):
            self._kv(l, a, pos)
        X = [list(self.h0) for _ in range(c.block)]
        hidden = []
        for l in range(c.n_layers):
            p = f"layers.{l}."
            n = 3 * l
            Hs = [lnmod(x, self.modpart(n, 0), self.modpart(n, 1), c.ln_eps) for x in X]
            qs, ks, vs = [], [], []
            for t, h in enumerate(Hs):
                pp = pos + 1 + t
                qs.append(headnorm_rope(matvec(self.W[p + "self_attn.q_proj.weight"], h),
                                        self.W[p + "self_attn.q_norm.weight"], c.qk_eps, hd, pp, c.rope_theta))
                ks.append(headnorm_rope(matvec(self.W[p + "self_attn.k_proj.weight"], h),
                                        self.W[p + "self_attn.k_norm.weight"], c.qk_eps, hd, pp, c.rope_theta))
                vs.append(matvec(self.W[p + "self_attn.v_proj.weight"], h))
            os_ = attend(qs, ks, vs, hd)
            g = self.modpart(n, 2)
            for t in range(c.block):
                y = matvec(self.W[p + "self_attn.o_proj.weight"], os_[t])
                X[t] = [X[t][i] + g[i] * y[i] for i in range(self.D)]
            n = 3 * l + 1
            Hs = [lnmod(x, self.modpart(n, 0), self.modpart(n, 1), c.ln_eps) for x in X]
            qs = [headnorm_rope(matvec(self.W[p + "cross_attn.q_proj.weight"], h),
                                self.W[p + "cross_attn.q_norm.weight"], c.qk_eps, hd, pos + 1 + t, c.rope_theta)
                  for t, h in enumerate(Hs)]
            ks = [self.K[l][r] for r in range(pos + 1)]
            vs = [self.V[l][r] for r in range(pos + 1)]
            os_ = attend(qs, ks, vs, hd)
            g = self.modpart(n, 2)
            for t in range(c.block):
                y = matvec(self.W[p + "cross_attn.o_proj.weight"], os_[t])
                X[t] = [X[t][i] + g[i] * y[i] for i in range(self.D)]
            n = 3 * l + 2
            g = self.modpart(n, 2)
            for t in range(c.block):
                h = lnmod(X[t], self.modpart(n, 0), self.modpart(n, 1), c.ln_eps)
                u = [gelu(v) for v in matvec(self.W[p + "mlp.fc1.weight"], h, self.W[p + "mlp.fc1.bias"])]
                y = matvec(self.W[p + "mlp.fc2.weight"], u, self.W[p + "mlp.fc2.bias"])
                X[t] = [X[t][i] + g[i] * y[i] for i in range(self.D)]
            hidden.append([list(x) for x in X])
        n = 3 * c.n_layers
        Y = [matvec(self.W["head.weight"], lnmod(x, self.modpart(n, 0), self.modpart(n, 1), c.ln_eps),
                    self.W["head.bias"]) for x in X]
        logits = [[sum(e[i] * y[i] for i in range(len(y))) for e in self.E] for y in Y]
        return [argmax(r) for r in logits], logits, Y, hidden


class BruteDFlash:
    def __init__(self, cfg, w):
        self.c = cfg
        self.W = {n: (mat(a) if a.ndim == 2 else vec(a)) for n, a in w.items()}
        self.E = self.W.pop("token_embd.weight")
        self.K = [dict() for _ in range(cfg.n_layers)]
        self.V = [dict() for _ in range(cfg.n_layers)]

    def append(self, feats, start):
        c = self.c
        for t, f in enumerate(feats):
            h = rmsn(vecmat([float(a) for a in f], self.W["W_c"]), self.W["ctx_norm"], c.rms_eps)
            for i in range(c.n_layers):
                nc = rmsn(h, self.W[f"bb.{i}.attn_norm"], c.rms_eps)
                self.K[i][start + t] = vecmat(nc, self.W[f"bb.{i}.k"])
                self.V[i][start + t] = vecmat(nc, self.W[f"bb.{i}.v"])

    def draft(self, anchor, pos):
        c = self.c
        W = self.W
        bp = W["block_pos"]
        a = vecmat(self.E[anchor], W["tok_proj"])
        Hd = [[a[i] + bp[0][i] for i in range(c.dim)]]
        for j in range(1, c.block):
            Hd.append([W["mask_emb"][j - 1][i] + bp[j][i] for i in range(c.dim)])
        hidden = []
        for i in range(c.n_layers):
            p = f"bb.{i}."
            nd = [rmsn(h, W[p + "attn_norm"], c.rms_eps) for h in Hd]
            qs = [vecmat(x, W[p + "q"]) for x in nd]
            kd = [vecmat(x, W[p + "k"]) for x in nd]
            vd = [vecmat(x, W[p + "v"]) for x in nd]
            ks = [self.K[i][r] for r in range(pos)] + kd
            vs = [self.V[i][r] for r in range(pos)] + vd
            os_ = attend(qs, ks, vs, c.head_dim)
            new = []
            for t in range(c.block):
                o = vecmat(os_[t], W[p + "o"])
                hcur = [Hd[t][j] + o[j] for j in range(c.dim)]
                n2 = rmsn(hcur, W[p + "ff_norm"], c.rms_eps)
                g = vecmat(n2, W[p + "gate"])
                u = vecmat(n2, W[p + "up"])
                m = vecmat([gelu_tanh(g[j]) * u[j] for j in range(len(g))], W[p + "down"])
                new.append([hcur[j] + m[j] for j in range(c.dim)])
            Hd = new
            hidden.append([list(h) for h in Hd])
        out = [rmsn(h, W["out_norm"], c.rms_eps) for h in Hd]
        Y = [vecmat(o, W["out_proj"]) for o in out]
        logits = [[sum(e[i] * y[i] for i in range(len(y))) for e in self.E] for y in Y]
        return [argmax(r) for r in logits], logits, Y, hidden


def time_conditioning(weights, n_layers: int, time_dim: int, time_scale: float, s: float, t: float):
    """flashmap_drafter.js ``timeConditioning`` by explicit loops: for each of
    s (time_embed) and t (jump_embed) a [cos | sin] embedding of width time_dim
    (frequencies exp(-ln(10000) i / half)), linear_1, x / (1 + exp(-x)),
    linear_2; cond = SiLU(sum); then every adaLN linear of cond, (self, cross,
    mlp) per layer and the final one."""
    def lin(name, x):
        W = mat(weights[name + ".weight"])
        b = vec(weights[name + ".bias"]) if name + ".bias" in weights else None
        return matvec(W, x, b)

    def sig_lu(v):
        return [x / (1.0 + math.exp(-x)) for x in v]

    def embed(prefix, time):
        half_ = time_dim // 2
        e = [0.0] * time_dim
        for i in range(half_):
            a = time * time_scale * math.exp(-math.log(10000.0) * i / half_)
            e[i] = math.cos(a)
            e[half_ + i] = math.sin(a)
        return lin(prefix + ".linear_2", sig_lu(lin(prefix + ".linear_1", e)))

    ts = embed("time_embed", s)
    tj = embed("jump_embed", t)
    cond = sig_lu([a + b for a, b in zip(ts, tj)])
    out = []
    for l in range(n_layers):
        for n in ("self_attn_adaln", "cross_attn_adaln", "mlp_adaln"):
            out.extend(lin(f"layers.{l}.{n}.linear", cond))
    out.extend(lin("final_adaln.linear", cond))
    return out


def dflash_sequential(weights, base_logits, block_rows, anchor: int, rms_eps: float, thresholds=None, min_conf=None):
    """The greedy sequential head by loops (module-dflash.ts ``forwardRows``):
    base_logits [gamma][V] and block_rows [gamma][d] (the backbone rows before
    out_norm) as lists; returns (tokens, conf, length)."""
    w1 = mat(weights["markov.w1"])
    rnn = "rnn.wH" in weights
    if rnn:
        wH, bH, wO = mat(weights["rnn.wH"]), vec(weights["rnn.bH"]), mat(weights["rnn.wO"])
    else:
        w2 = mat(weights["markov.w2"])
    onw = vec(weights["out_norm"])
    cw = [row[0] for row in mat(weights["conf.w"])] if "conf.w" in weights else None
    cb = vec(weights["conf.b"])[0] if "conf.b" in weights else 0.0
    r = len(w1[0])
    V = len(base_logits[0])
    s = [0.0] * r
    prev = anchor
    tokens, conf = [], []
    for k in range(len(base_logits)):
        e1 = w1[prev]
        if rnn:
            s = [math.tanh(sum(s[i] * wH[i][j] for i in range(r)) + e1[j] + bH[j]) for j in range(r)]
            bias = [sum(s[i] * wO[i][v] for i in range(r)) for v in range(V)]
        else:
            bias = [sum(e1[i] * w2[i][v] for i in range(r)) for v in range(V)]
        sc = [base_logits[k][v] + bias[v] for v in range(V)]
        best = 0
        for v in range(1, V):
            if sc[v] > sc[best]:
                best = v
        tokens.append(best)
        prev = best
        if cw is not None:
            row = block_rows[k]
            ms = sum(x * x for x in row) / len(row)
            h = [row[i] * onw[i] / math.sqrt(ms + rms_eps) for i in range(len(row))]
            z = sum(a * b for a, b in zip(h + list(e1), cw)) + cb
            conf.append(1.0 / (1.0 + math.exp(-z)))
            thr = None
            if thresholds is not None and k < len(thresholds) and thresholds[k] is not None and thresholds[k] == thresholds[k]:
                thr = thresholds[k]
            if thr is None:
                thr = min_conf
            if k > 0 and thr is not None and conf[-1] < thr:
                return tokens, conf, k
    return tokens, conf, len(tokens)


def mtp_forward(weights, cfg, tokens, hn_rows, pos0: int, kv_lo: int, kcache, vcache):
    """The MTP head's forward over len(tokens) rows by loops (ternary_bonsai_2_mtp.js,
    ``MTPHead.forward`` and its WGSL kernels); kcache / vcache are lists of rows
    (None where unwritten), updated in place.  Returns the shared_head_norm rows."""
    H, hd, nh, nkv, rot, eps = cfg.hidden, cfg.head_dim, cfg.n_heads, cfg.n_kv_heads, cfg.rot_dims, cfg.eps
    Wm = {n: [q8_row(r, k) for r in weights[n]] for n, k in (
        ("eh_proj", 2 * H), ("attn_q", H), ("attn_k", H), ("attn_v", H), ("attn_output", nh * hd),
        ("ffn_gate", H), ("ffn_up", H), ("ffn_down", cfg.inter))}
    nw = {n: [float(v) for v in weights[n]] for n in ("enorm", "hnorm", "attn_norm", "attn_q_norm", "attn_k_norm",
                                                    "post_attention_norm", "shared_head_norm")}

    def rope(y, pos):
        y = list(y)
        half_ = rot // 2
        for i in range(half_):
            ang = pos * theta_pow(i)
            c, s = math.cos(ang), math.sin(ang)
            a0, a1 = y[i], y[i + half_]
            y[i] = a0 * c - a1 * s
            y[i + half_] = a1 * c + a0 * s
        return y

    def theta_pow(i):
        return cfg.theta ** (-2.0 * i / rot)

    rows = []
    for m, tok in enumerate(tokens):
        e = [bf(b) for b in weights["token_embd"][tok]]
        xc = rmsn(e, nw["enorm"], eps) + rmsn([float(v) for v in hn_rows[m]], nw["hnorm"], eps)
        x = matvec(Wm["eh_proj"], xc)
        a = rmsn(x, nw["attn_norm"], eps)
        qf = matvec(Wm["attn_q"], a)
        kt = matvec(Wm["attn_k"], a)
        vt = matvec(Wm["attn_v"], a)
        pos = pos0 + m
        krow, vrow = [], []
        for g in range(nkv):
            krow += rope(rmsn(kt[g * hd:(g + 1) * hd], nw["attn_k_norm"], eps), pos)
        kcache[pos] = krow
        vcache[pos] = list(vt)
        rows.append((x, qf, pos))
    outs = []
    for x, qf, pos in rows:
        gated = []
        for h in range(nh):
            q = rope(rmsn(qf[h * 2 * hd:h * 2 * hd + hd], nw["attn_q_norm"], eps), pos)
            g = h // (nh // nkv)
            sc = []
            for j in range(kv_lo, pos + 1):
                s = 0.0
                for d in range(hd):
                    s += q[d] * kcache[j][g * hd + d]
                sc.append(s / math.sqrt(hd))
            mx = max(sc)
            es = [math.exp(s - mx) for s in sc]
            tot = sum(es)
            for d in range(hd):
                acc = 0.0
                for jj, j in enumerate(range(kv_lo, pos + 1)):
                    acc += es[jj] * vcache[j][g * hd + d]
                gate = qf[h * 2 * hd + hd + d]
                gated.append(acc / tot / (1.0 + math.exp(-gate)))
        o = matvec(Wm["attn_output"], gated)
        x = [x[i] + o[i] for i in range(H)]
        a = rmsn(x, nw["post_attention_norm"], eps)
        gt = matvec(Wm["ffn_gate"], a)
        up = matvec(Wm["ffn_up"], a)
        f = [gt[i] / (1.0 + math.exp(-gt[i])) * up[i] for i in range(len(gt))]
        dn = matvec(Wm["ffn_down"], f)
        x = [x[i] + dn[i] for i in range(H)]
        outs.append(rmsn(x, nw["shared_head_norm"], eps))
    return outs
