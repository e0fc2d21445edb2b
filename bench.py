#!/usr/bin/env python
"""Benchmark of the drafter hot path on GB300.

Default workload (N = 1): the FlashMap-Qwen3-4B-shaped draft step --
fm_context_append of 17 feature rows at position 1024 (rewinding to 1024 every
step, so every step is identical) followed by fm_draft of the 16-slot block at
position 1041 (1042 cross-attention keys).  One step reads ~1.3 GB (all
weights, the Q8_0 table, the cache), far more than the 129 MB L2, so no L2
flush is needed between steps.

Prints one JSON line.  ``--impl reference`` times the CPU oracle (the only
reference implementation of this path) on the same workload.
``--workload`` selects another configuration's timed unit: prefill (32768-row
context injection, then a draft over 32769 keys), dflash (draft / append
cycles), batched (32 sequences), tiny.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft steps/sec + achieved HBM GB/s (16-slot block); context prefill rows/sec"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="flashmap4b", choices=["flashmap4b", "prefill", "dflash", "dflash_seq", "tiny", "batched", "mtp"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true", help="skip the secondary prefill rows/s figure")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    p.add_argument("--no-kprof", action="store_true", help="skip the per-kernel timing pass")
    p.add_argument("--prefill-rows", type=int, default=32768, help="rows of the prefill workload (a smaller case "
                   "for profiling captures)")
    p.add_argument("--batched-ctx", type=int, default=8192, help="longest context of the batched workload (a "
                   "smaller case for profiling captures; contexts are uniform in [512, this])")
    return p.parse_args()


# ----------------------------------------------------------------- helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), float(m.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# kernel tag (as fm_profile_read names it) -> the source file that defines it
KERNEL_SOURCES = {"lm_head": ("k_lmhead.cu",), "attn": ("k_attn.cu",), "gemv": ("k_gemv.cu", "linear_parts.cuh"),
                  "seq": ("k_seqhead.cu",), "draft_step": ("k_step.cu", "linear_parts.cuh"),
                  "prefill": ("k_gemm.cu", "tc_gemm.h"), "append": ("k_gemm.cu", "tc_gemm.h"),
                  "wide": ("k_gemm.cu", "tc_gemm.h", "k_wide.cu", "k_xattn.cu")}


def source_digest(tag):
    """Digest of the sources the kernel behind `tag` is built from: its own
    files and the two headers every kernel includes."""
    import hashlib
    src = KERNEL_SOURCES.get(tag.split(".")[0])
    if src is None:
        return None
    h = hashlib.sha256()
    for name in (*src, "dev_common.cuh", "fm_internal.h"):
        with open(os.path.join(ROOT, "block_speculative_decoding_fm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


WORKLOAD = "flashmap4b"   # the workload of this run (a kernel tag's traffic depends on it)


def ncu_traffic(tag):
    """DRAM bytes (read + write) per launch of the kernel behind `tag` in this
    run's workload, from the committed ncu summary profiles/ncu_dram_traffic.txt
    (lines `tag@workload`, or a bare `tag` for the default FlashMap-4B step), or
    None when there is no capture or the kernel's sources have changed since it
    was taken (each line records source_digest() of the build the capture ran)."""
    digest = source_digest(tag)
    path = os.path.join(ROOT, "profiles", "ncu_dram_traffic.txt")
    if digest is None or not os.path.exists(path):
        return None
    names = {f"{tag}@{WORKLOAD}"} | ({tag} if WORKLOAD == "flashmap4b" else set())
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] in names and parts[3] == digest:
                return float(parts[1])
    return None


class Clocks:
    """nvidia-smi samples every 50 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier_max(ws, value, device="cuda"):
    """The largest of the ranks' values (the slowest rank's time): every rank gets it."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as d
    t = torch.tensor([value], dtype=torch.float64, device=device)
    d.all_reduce(t, op=d.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(steps, ws, ms):
    """Units per second of the whole job: every rank ran `steps` units; ms is the slowest rank's time."""
    return steps * ws / (ms / 1000)


# ----------------------------------------------------------------- workloads

class FlashMapStep:
    """append(17 rows at 1024) + draft(anchor, 1041) on the FlashMap-4B shape."""
    name = "flashmap4b_step"

    def __init__(self, torch):
        import block_speculative_decoding_fm_gb300 as fm
        import fm_synth as S
        self.fm, self.S, self.torch = fm, S, torch
        self.cfg = S.flashmap_4b_config()
        w = S.gen_weights(self.cfg, 1002)
        self.mod = S.gen_modulation(self.cfg, 1002)
        self.h = fm.fm_create(self.cfg, fm.weight_items(w), self.mod)
        self.raw = {n: t.data for n, t in w.items()}
        fr = S.streams(1002)["features"]
        self.ctx = S.gen_features(fr, 1024, self.cfg.feat_dim)
        self.f17 = S.gen_features(fr, 17, self.cfg.feat_dim)
        self.anchor = S.gen_anchor(S.streams(1002)["tokens"], self.cfg.vocab)
        fm.fm_context_append(self.h, 0, torch.from_numpy(self.ctx).cuda(), 1024, 0)
        self.f17_dev = torch.from_numpy(self.f17).cuda()
        self.tokens = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
        self.f17_host = torch.from_numpy(self.f17).pin_memory()
        self.tok_host = torch.zeros((1, 16), dtype=torch.int32).pin_memory()
        self.launches = 0
        c = self.cfg
        D, F, Ht, L = c.dim, c.ff_dim, c.target_dim, c.n_layers
        weights = (D * c.feat_dim + D * Ht * 2 + L * (4 * D * D + 4 * D * D + 2 * F * D) + Ht * D) * 2
        table = c.vocab * (Ht + Ht // 16)
        kv_read = L * 2 * 1042 * D * 2
        feats = 17 * c.feat_dim * 4
        kv_write = L * 2 * 18 * D * 2
        self.bytes_per_step = weights + table + kv_read + feats + kv_write
        # the anchor row's K/V projection re-reads the 12 cross K/V matrices
        self.bytes_per_step_moved = self.bytes_per_step + L * 2 * D * D * 2

    def step(self):
        fm = self.fm
        fm.fm_context_append(self.h, 0, self.f17_dev, 17, 1024)
        self.launches += fm.fm_last_launch_count(self.h)
        fm.fm_draft(self.h, [0], [self.anchor], [1041], self.tokens)
        self.launches += fm.fm_last_launch_count(self.h)

    def step_e2e(self):
        # the host-buffer calls of the C ABI: rows copied in, tokens copied out, on the stream
        fm = self.fm
        fm.fm_context_append_host(self.h, 0, self.f17_host, 17, 1024)
        self.launches += fm.fm_last_launch_count(self.h)
        fm.fm_draft_host(self.h, [0], [self.anchor], [1041], self.tok_host)
        self.launches += fm.fm_last_launch_count(self.h)

    e2e_h2d = 17 * 12800 * 4
    e2e_d2h = 16 * 4

    def oracle_setup(self):
        from oracle import FlashMap
        o = FlashMap(self.cfg, self.raw, self.mod, True)
        st = o.new_state()
        o.context_append(st, self.ctx, 0)
        return o, st

    def oracle_step(self, o, st):
        o.context_append(st, self.f17, 1024)
        o.draft(st, self.anchor, 1041)


class PrefillStep:
    """fm_context_append of 32768 feature rows (12800 wide) from position 0."""
    name = "prefill_32768"

    def __init__(self, torch, rows=32768):
        import block_speculative_decoding_fm_gb300 as fm
        import fm_synth as S
        self.fm, self.torch, self.rows = fm, torch, rows
        self.cfg = S.flashmap_4b_config(max_ctx=rows + 64)
        w = S.gen_weights(self.cfg, 1003)
        self.h = fm.fm_create(self.cfg, fm.weight_items(w), S.gen_modulation(self.cfg, 1003))
        self.feats = torch.from_numpy(S.gen_features(S.streams(1003)["features"], rows, self.cfg.feat_dim)).cuda()
        self.launches = 0
        c = self.cfg
        self.flops = 2.0 * rows * c.dim * (c.feat_dim + 2 * c.n_layers * c.dim)

    def step(self):
        self.fm.fm_context_append(self.h, 0, self.feats, self.rows, 0)
        self.launches += self.fm.fm_last_launch_count(self.h)


class TinyStep:
    """Config 1: the tiny drafter, 64 context rows; one timed unit = draft at 64 + device acceptance."""
    name = "tiny_step"

    def __init__(self, torch):
        import block_speculative_decoding_fm_gb300 as fm
        import fm_synth as S
        self.fm, self.torch = fm, torch
        self.cfg = S.tiny_config(max_ctx=128)
        w = S.gen_weights(self.cfg, 1001)
        self.h = fm.fm_create(self.cfg, fm.weight_items(w), S.gen_modulation(self.cfg, 1001))
        fm.fm_context_append(self.h, 0, torch.from_numpy(S.gen_features(S.streams(1001)["features"], 64,
                                                                       self.cfg.feat_dim)).cuda(), 64, 0)
        self.anchor = S.gen_anchor(S.streams(1001)["tokens"], self.cfg.vocab)
        self.tokens = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
        self.target = torch.zeros((1, 17), dtype=torch.int32, device="cuda")
        self.k = torch.full((1,), 16, dtype=torch.int32, device="cuda")
        self.acc = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.bonus = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.launches = 0

    def step(self):
        fm = self.fm
        fm.fm_draft(self.h, [0], [self.anchor], [64], self.tokens)
        self.launches += fm.fm_last_launch_count(self.h)
        fm.fm_accept_batched(self.h, self.tokens, self.target, self.k, self.acc, self.bonus)
        self.launches += 1


class DFlashCycles:
    """Config 4: the DFlash drafter, 4096 context rows, then draft -> accept -> append acc + 1 rows at the
    anchor position, with seeded acceptance counts in [0, 5]; one timed unit = one cycle.  seq_head: the
    drafter also carries the Markov sequential head (rank 256) and the confidence head, and drafts through
    fm_draft_pruned with a uniform min_conf."""
    name = "dflash_cycle"

    def __init__(self, torch, cycles, seq_head=False):
        import block_speculative_decoding_fm_gb300 as fm
        import fm_synth as S
        self.fm, self.torch = fm, torch
        self.cfg = S.dflash_config(max_ctx=4096 + 6 * cycles + 64)
        c = self.cfg
        w = S.gen_weights(self.cfg, 1004)
        self.seq_head = seq_head
        if seq_head:
            w.update(S.gen_seq_head_weights(self.cfg, 1004, "markov", rank=256))
            self.conf = torch.zeros((c.block,), dtype=torch.float32, device="cuda")
            self.length = torch.zeros((1,), dtype=torch.int32, device="cuda")
        self.h = fm.fm_create(self.cfg, fm.weight_items(w), S.gen_modulation(self.cfg, 1004))
        g = torch.Generator(device="cuda")
        g.manual_seed(1004)
        ctx = torch.randn((4096, c.feat_dim), generator=g, device="cuda")
        fm.fm_context_append(self.h, 0, ctx, 4096, 0)
        del ctx
        self.pool = torch.randn((6 * cycles + 6, c.feat_dim), generator=g, device="cuda")
        rng = np.random.default_rng(1004)
        self.acc = rng.integers(0, c.block + 1, size=cycles + 8)
        self.anchors = rng.integers(0, c.vocab, size=cycles + 8)
        self.tokens = torch.zeros((1, c.block), dtype=torch.int32, device="cuda")
        self.pos, self.i, self.used, self.launches = 4096, 0, 0, 0
        table = c.vocab * c.target_dim * 2
        seq = ("markov.", "rnn.", "conf.")
        others = sum(t.data.nbytes for n, t in w.items() if not n.startswith(seq)) - table
        self.bytes_fixed = table + others
        if seq_head:
            # per position: markov.w2 streamed once, the base logits row read; the lm_head stores the rows
            self.bytes_fixed += c.block * (256 * c.vocab * 2 + c.vocab * 4) + c.block * c.vocab * 4

    def bytes_at(self, pos):
        c = self.cfg
        return self.bytes_fixed + c.n_layers * 2 * pos * c.dim * 2

    def step(self):
        fm = self.fm
        if self.seq_head:
            fm.fm_draft_pruned(self.h, 0, int(self.anchors[self.i]), self.pos, self.tokens[0], self.conf,
                               self.length, min_conf=0.5)
        else:
            fm.fm_draft(self.h, [0], [int(self.anchors[self.i])], [self.pos], self.tokens)
        self.launches += fm.fm_last_launch_count(self.h)
        n = int(self.acc[self.i]) + 1
        fm.fm_context_append(self.h, 0, self.pool[self.used:self.used + n], n, self.pos)
        self.launches += fm.fm_last_launch_count(self.h)
        self.pos += n
        self.used += n
        self.i += 1


class MtpCycle:
    """The MTP draft head at the page's MCFG shape (Q8_0 layer, vocab 248,320): a draft of depth 3 from two
    pending rows (a 2-row pass, then two chained single-row passes on the device's own drafts) over a
    1,024-row head cache; one timed unit = one draft.  The pending rows re-write the same cache rows every
    step."""
    name = "mtp_draft"

    def __init__(self, torch, depth=3, history=1024):
        import block_speculative_decoding_fm_gb300 as fm
        import fm_synth as S
        self.fm, self.torch, self.depth = fm, torch, depth
        self.cfg = c = S.mtp_config(kv_cap=history + 64)
        self.w = S.gen_mtp_weights(c, 1206)
        self.h = fm.fm_mtp_create(c, fm.weight_items(self.w))
        g = torch.Generator(device="cuda")
        g.manual_seed(1206)
        for p0 in range(0, history, 8):
            toks = torch.randint(0, c.vocab, (8,), generator=g, device="cuda", dtype=torch.int32)
            fm.fm_mtp_forward(self.h, toks, torch.randn((8, c.hidden), generator=g, device="cuda"), p0, 0)
        self.pos = history
        self.toks = torch.randint(0, c.vocab, (2,), generator=g, device="cuda", dtype=torch.int32)
        self.hn = torch.randn((2, c.hidden), generator=g, device="cuda")
        self.drafts = torch.zeros((depth,), dtype=torch.int32, device="cuda")
        self.launches = 0
        q8 = lambda n, k: n * k // 32 * 34
        H, I, nh, nkv, hd = c.hidden, c.inter, c.n_heads, c.n_kv_heads, c.head_dim
        layer = (q8(H, 2 * H) + q8(nh * 2 * hd + 2 * nkv * hd, H) + q8(H, nh * hd) + q8(2 * I, H) + q8(H, I)
                 + 7 * H * 4 + 2 * hd * 4)
        lm = q8(c.vocab, H)
        cache = (history + 2) * 2 * nkv * hd * 4
        # per pass: the layer's weights, the lm_head table and the head cache rows it attends over (read once)
        self.bytes_per_step = depth * (layer + lm + cache)

    def step(self):
        fm = self.fm
        fm.fm_mtp_draft(self.h, self.toks, self.hn, self.pos, 0, self.depth, self.drafts)
        self.launches += fm.fm_mtp_last_launch_count(self.h)


class BatchedStep:
    """Config 5: 32 sequences, contexts U[512, 8192] (prefilled untimed), each appends acc_i + 1 rows
    (acc_i ~ U{0..16}) then all 32 draft 16 slots; every step re-appends at the same positions."""
    name = "batched_32_step"

    def __init__(self, torch, n_seqs=32, ctx_hi=8192):
        import block_speculative_decoding_fm_gb300 as fm
        import fm_synth as S
        self.fm, self.torch = fm, torch
        self.cfg = S.flashmap_4b_config(max_ctx=ctx_hi + 17 + 64, max_seqs=n_seqs)
        c = self.cfg
        w = S.gen_weights(self.cfg, 1005)
        self.h = fm.fm_create(self.cfg, fm.weight_items(w), S.gen_modulation(self.cfg, 1005))
        rng = S.streams(1005)["workload"]
        self.L = [int(x) for x in S.batched_lengths(rng, n_seqs, hi=ctx_hi)]
        self.n = [int(x) + 1 for x in rng.integers(0, 17, size=n_seqs)]
        self.anchors = [int(x) for x in rng.integers(0, c.vocab, size=n_seqs)]
        g = torch.Generator(device="cuda")
        g.manual_seed(1005)
        for i, L in enumerate(self.L):
            f = torch.randn((L, c.feat_dim), generator=g, device="cuda")
            fm.fm_context_append(self.h, i, f, L, 0)
            del f
        self.feats = torch.randn((sum(self.n), c.feat_dim), generator=g, device="cuda")
        self.ids = list(range(n_seqs))
        self.pos = [L + n for L, n in zip(self.L, self.n)]
        self.tokens = torch.zeros((n_seqs, 16), dtype=torch.int32, device="cuda")
        self.feats_host = self.feats.cpu().pin_memory()
        self.tok_host = torch.zeros((n_seqs, 16), dtype=torch.int32).pin_memory()
        self.e2e_h2d = sum(self.n) * c.feat_dim * 4
        self.e2e_d2h = n_seqs * 16 * 4
        self.launches = 0
        D, F, Ht, Ll = c.dim, c.ff_dim, c.target_dim, c.n_layers
        weights = (D * c.feat_dim + D * Ht * 2 + Ll * (4 * D * D + 4 * D * D + 2 * F * D) + Ht * D) * 2
        table = c.vocab * (Ht + Ht // 16)
        kv = sum((p + 1) * Ll * 2 * D * 2 for p in self.pos)
        self.bytes_per_step = weights + table + kv + sum(self.n) * c.feat_dim * 4

    def step(self):
        fm = self.fm
        fm.fm_context_append_batched(self.h, self.ids, self.feats, self.n, self.L)
        self.launches += fm.fm_last_launch_count(self.h)
        fm.fm_draft(self.h, self.ids, self.anchors, self.pos, self.tokens)
        self.launches += fm.fm_last_launch_count(self.h)

    def step_e2e(self):
        fm = self.fm
        fm.fm_context_append_batched_host(self.h, self.ids, self.feats_host, self.n, self.L)
        self.launches += fm.fm_last_launch_count(self.h)
        fm.fm_draft_host(self.h, self.ids, self.anchors, self.pos, self.tok_host)
        self.launches += fm.fm_last_launch_count(self.h)


def kernel_profile(fm, h, step, n):
    """Per-kernel device time over n steps (FM_DEBUG_PROFILE brackets every
    launch with CUDA events on its stream): {name: (launches, ms, bytes)}."""
    fm.fm_set_debug(h, fm.FM_DEBUG_PROFILE)
    for _ in range(n):
        step()
    prof = fm.fm_profile_read(h)
    fm.fm_set_debug(h, 0)
    return prof


def hbm_roofline(prof, hbm, peak_src, steps):
    """The kernel with the largest device time per step against the HBM copy peak."""
    name, (nl, tms, tb) = max(prof.items(), key=lambda kv: kv[1][1])
    achieved = (tb / nl) / ((tms / nl) / 1000) / 1e9
    return {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": ncu_traffic(name), "peak_source": f"{peak_src} burst copy", "bytes_per_launch": tb / nl,
            "ms_per_launch": tms / nl}, \
        {k: {"launches": v[0] / steps, "ms_per_step": v[1] / steps} for k, v in sorted(prof.items())}


def dominant_roofline(prof, hbm, bf16_sustained, peak_src, steps):
    """The kernel with the largest device time per step against its own bound:
    the tensor-core GEMMs (names holding "gemm", whose records carry FLOPs)
    against the sustained bf16 peak (timed inside a long step), the rest
    against the HBM copy peak."""
    name, (nl, tms, tq) = max(prof.items(), key=lambda kv: kv[1][1])
    kernels = {k: {"launches": v[0] / steps, "ms_per_step": v[1] / steps} for k, v in sorted(prof.items())}
    if "gemm" not in name:
        return hbm_roofline(prof, hbm, peak_src, steps)[0], kernels
    achieved = (tq / nl) / ((tms / nl) / 1000) / 1e12
    return {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": bf16_sustained, "unit": "TFLOP/s",
            "frac": achieved / bf16_sustained, "traffic": ncu_traffic(name),
            "peak_source": f"{peak_src} bf16 sustained (f16 has the same nominal tensor rate)",
            "flops_per_launch": tq / nl, "ms_per_launch": tms / nl}, kernels


def oracle_sample(fn, budget_s=15.0, most=20):
    """Run fn() until the budget or `most` repetitions; (repetitions, seconds)."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= most:
            break
    return n, time.perf_counter() - t0


def run_workload(args):
    """The other configs' timed units (one JSON line each, same keys as the default line)."""
    import torch
    torch.cuda.set_device(0)
    from block_speculative_decoding_fm_gb300 import build
    build.build()
    import block_speculative_decoding_fm_gb300 as fm
    import fm_synth as S
    hbm, bf16, bf16s, peak_src = peaks()
    cores = len(os.sched_getaffinity(0))
    extra, unit, value, ms, launches = {}, "steps/s", None, None, 0
    roofline, kernels, cpu, e2e = None, None, None, None
    with Clocks(0) as clk:
        if args.workload == "tiny":
            w = TinyStep(torch)
            for _ in range(max(3, args.warmup)):
                w.step()
            w.launches = 0
            ms = time_steps(torch, w.step, args.steps)
            value, launches = args.steps / (ms / 1000), w.launches
            cfgd = {"workload": "tiny: D 256, 2 layers, 64 context rows, draft at 64 + device acceptance"}
        elif args.workload in ("dflash", "dflash_seq"):
            # cycles for the warm-up, the timed steps and the per-kernel pass below
            w = DFlashCycles(torch, args.steps + max(3, args.warmup) + 20 + 8, seq_head=args.workload == "dflash_seq")
            for _ in range(max(3, args.warmup)):
                w.step()
            w.launches = 0
            p0 = w.pos
            ms = time_steps(torch, w.step, args.steps)
            value, unit, launches = args.steps / (ms / 1000), "cycles/s", w.launches
            gb = (w.bytes_at(p0) + w.bytes_at(w.pos)) / 2 * args.steps / 1e9
            extra["achieved_hbm_gbs"] = gb / (ms / 1000)
            extra["bytes_per_cycle"] = (w.bytes_at(p0) + w.bytes_at(w.pos)) / 2
            cfgd = {"workload": f"dflash: D 1024, 5 layers, gamma 5, bf16 vocab 262144, context {p0}..{w.pos} "
                                "(draft -> append acc+1 rows, acc seeded in [0,5])"}
            if w.seq_head:
                cfgd["workload"] += "; Markov sequential head rank 256 + confidence pruning at min_conf 0.5"
        elif args.workload == "mtp":
            w = MtpCycle(torch)
            for _ in range(max(3, args.warmup)):
                w.step()
            w.launches = 0
            ms = time_steps(torch, w.step, args.steps)
            value, unit, launches = args.steps / (ms / 1000), "drafts/s", w.launches
            extra["achieved_hbm_gbs"] = w.bytes_per_step * value / 1e9
            extra["bytes_per_step"] = w.bytes_per_step
            extra["tokens_drafted_per_s"] = value * w.depth
            cfgd = {"workload": "mtp: MTP head H 5120, I 17408, 24/4 heads x 256, Q8_0, vocab 248320; depth-3 draft "
                                "from 2 pending rows over a 1024-row head cache"}
        elif args.workload == "batched":
            w = BatchedStep(torch, ctx_hi=args.batched_ctx)
            for _ in range(max(3, args.warmup)):
                w.step()
            w.launches = 0
            ms = time_steps(torch, w.step, args.steps)
            value, launches = args.steps / (ms / 1000), w.launches
            extra["tokens_drafted_per_s"] = value * 32 * 16
            extra["achieved_hbm_gbs"] = w.bytes_per_step * value / 1e9
            extra["bytes_per_step"] = w.bytes_per_step
            if not args.no_e2e:
                # the host-buffer calls: the step's feature rows in, the drafted tokens out, inside the timed region
                for _ in range(3):
                    w.step_e2e()
                ms_e2e = time_steps(torch, w.step_e2e, args.steps)
                e2e = {"value": args.steps / (ms_e2e / 1000), "unit": "steps/s", "h2d_bytes_per_step": w.e2e_h2d,
                       "d2h_bytes_per_step": w.e2e_d2h}
            cfgd = {"workload": f"batched: 32 FlashMap-4B sequences, contexts U[512,{args.batched_ctx}], append "
                                "acc_i+1 rows (acc_i in 0..16) + 32 x 16-slot draft", "global_batch": 512}
        else:   # prefill
            w = PrefillStep(torch, rows=args.prefill_rows)
            w.step()
            torch.cuda.synchronize()
            w.launches = 0
            n = max(10, args.steps // 20)
            ms = time_steps(torch, w.step, n)
            value, unit, launches = w.rows * n / (ms / 1000), "rows/s", w.launches
            extra["prefill_tflops"] = w.flops * n / (ms / 1000) / 1e12
            extra["tensor_frac_of_measured_bf16"] = extra["prefill_tflops"] / bf16
            extra["prefill_reps"] = n
            # then the 16-slot draft over the 32768-row context (L = 32769)
            tok = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
            fm.fm_draft(w.h, [0], [123], [w.rows], tok)
            dms = time_steps(torch, lambda: fm.fm_draft(w.h, [0], [123], [w.rows], tok), 10) / 10
            torch.cuda.synchronize()
            extra["draft_after_prefill_ms"] = dms
            ms = ms * args.steps / n   # reported per the requested steps below
            cfgd = {"workload": f"prefill: fm_context_append of {w.rows} rows x 12800 (FlashMap-4B), then a draft at "
                                f"L={w.rows + 1}"}
    # per-kernel device times (a separate pass) and the roofline of the dominant kernel
    if args.workload == "prefill":
        prof = kernel_profile(fm, w.h, w.step, 3)
        gemm = [(k, v) for k, v in prof.items() if k.startswith("prefill.gemm")]
        flops = sum(v[2] for _, v in gemm)
        gms = sum(v[1] for _, v in gemm)
        achieved = flops / (gms / 1000) / 1e12
        roofline = {"bound": "tensor", "kernel": "prefill.gemm_fc + prefill.gemm_kv (tcgen05, f16 operands)",
                    "achieved": achieved, "peak": bf16, "unit": "TFLOP/s", "frac": achieved / bf16, "traffic": None,
                    "peak_source": f"{peak_src} bf16 burst (f16 has the same nominal tensor rate)",
                    "flops_per_launch": flops / max(1, sum(v[0] for _, v in gemm)),
                    "ms_per_launch": gms / max(1, sum(v[0] for _, v in gemm))}
        kernels = {k: {"launches": v[0] / 3, "ms_per_step": v[1] / 3} for k, v in sorted(prof.items())}
    elif args.workload == "batched":
        # the batched pass is one serial chain: per-kernel events; the dominant kernel against its own bound
        prof = kernel_profile(fm, w.h, w.step, 5)
        roofline, kernels = dominant_roofline(prof, hbm, bf16s or bf16, peak_src, 5)
        gemm = [v for k, v in prof.items() if "gemm" in k]
        if gemm:
            extra["gemm_tflops"] = sum(v[2] for v in gemm) / (sum(v[1] for v in gemm) / 1000) / 1e12
            extra["gemm_ms_per_step"] = sum(v[1] for v in gemm) / 5
        if "wide.attn_cross" in prof:
            v = prof["wide.attn_cross"]
            extra["attn_cross_gbs"] = v[2] / (v[1] / 1000) / 1e9
            extra["attn_cross_ms_per_step"] = v[1] / 5
    elif args.workload == "mtp":
        # the head's launches are not profiled one by one: the roofline of the whole step
        achieved = extra["achieved_hbm_gbs"]
        roofline = {"bound": "hbm", "kernel": f"{w.name} (every launch of the step)", "achieved": achieved,
                    "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                    "peak_source": f"{peak_src} burst copy", "bytes_per_launch": w.bytes_per_step,
                    "ms_per_launch": ms / args.steps}
    elif args.workload != "tiny":
        steps = 5 if args.workload == "batched" else 20
        roofline, kernels = hbm_roofline(kernel_profile(fm, w.h, w.step, steps), hbm, peak_src, steps)
    # the oracle on a bounded sample of the same workload, on the host cores
    if not args.no_cpu_baseline:
        from oracle import DFlash, FlashMap
        if args.workload == "prefill":
            c = w.cfg
            o = FlashMap(c, {n_: t.data for n_, t in S.gen_weights(c, 1003).items()}, S.gen_modulation(c, 1003), True)
            st = o.new_state(1024)
            rows = S.gen_features(S.streams(1003)["features"], 256, c.feat_dim)
            k, dt = oracle_sample(lambda: o.context_append(st, rows, 0), 15.0, 10)
            cpu = {"value": 256 * k / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
                   "sample": f"{k} appends of 256 of the 32768 rows in {dt:.1f} s", "blas_threads": blas_threads()}
        elif args.workload in ("dflash", "dflash_seq"):
            c = S.dflash_config(max_ctx=4096 + 64)
            wd = S.gen_weights(c, 1004)
            if args.workload == "dflash_seq":
                wd.update(S.gen_seq_head_weights(c, 1004, "markov", rank=256))
            o = DFlash(c, {n_: t.data for n_, t in wd.items()})
            del wd
            st = o.new_state()
            fr = S.streams(1004)["features"]
            o.context_append(st, S.gen_features(fr, 4096, c.feat_dim), 0)
            row = S.gen_features(fr, 1, c.feat_dim)

            def cycle():   # draft at the context length, then append one row at the anchor position
                pos = st.length
                res = o.draft(st, 7, pos)
                if args.workload == "dflash_seq":
                    o.sequential_head(res, 7, min_conf=0.5)
                o.context_append(st, row, pos)
            k, dt = oracle_sample(cycle, 15.0, 10)
            cpu = {"value": k / dt, "unit": "cycles/s", "cores": cores, "kind": "oracle",
                   "sample": f"{k} draft + 1-row append cycles at context 4096 in {dt:.1f} s",
                   "blas_threads": blas_threads()}
        elif args.workload == "mtp":
            from oracle.mtp import MtpHead
            c = w.cfg
            o = MtpHead(c, {n_: t.data for n_, t in w.w.items()})
            st = o.new_state()
            rng = S.streams(1206)["features"]
            o.forward(st, o.embed(list(range(8))), S.gen_mtp_hidden(rng, 8, c.hidden).astype(np.float64), 0, 0)
            hn = S.gen_mtp_hidden(rng, 2, c.hidden).astype(np.float64)
            k, dt = oracle_sample(lambda: o.draft(st, [5, 6], hn, 8, 0, 3), 20.0, 3)
            cpu = {"value": k / dt, "unit": "drafts/s", "cores": cores, "kind": "oracle",
                   "sample": f"{k} depth-3 drafts over an 8-row head cache in {dt:.1f} s (fp64, lm_head dequantised "
                             "by row blocks)", "blas_threads": blas_threads()}
        elif args.workload == "batched":
            c = S.flashmap_4b_config(max_ctx=4096 + 64)
            o = FlashMap(c, {n_: t.data for n_, t in S.gen_weights(c, 1005).items()}, S.gen_modulation(c, 1005), True)
            st = o.new_state()
            fr = S.streams(1005)["features"]
            o.context_append(st, S.gen_features(fr, 4352, c.feat_dim)[:4080], 0)
            rows = S.gen_features(fr, 9, c.feat_dim)
            k, dt = oracle_sample(lambda: (o.context_append(st, rows, 4080), o.draft(st, 7, 4089)), 15.0, 10)
            cpu = {"value": k / dt / 32, "unit": "steps/s", "cores": cores, "kind": "oracle",
                   "sample": f"{k} single-sequence append (9 rows) + draft at the mean context 4089 in {dt:.1f} s, "
                             "scaled to 32 sequences", "blas_threads": blas_threads()}
        else:
            c = S.tiny_config(max_ctx=128)
            o = FlashMap(c, {n_: t.data for n_, t in S.gen_weights(c, 1001).items()}, S.gen_modulation(c, 1001), False)
            st = o.new_state()
            o.context_append(st, S.gen_features(S.streams(1001)["features"], 64, c.feat_dim), 0)
            k, dt = oracle_sample(lambda: o.draft(st, 7, 64), 10.0, 200)
            cpu = {"value": k / dt, "unit": "steps/s", "cores": cores, "kind": "oracle",
                   "sample": f"{k} drafts in {dt:.1f} s", "blas_threads": blas_threads()}
    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfgd, "e2e": e2e,
            "gpu_launches": launches, "roofline": roofline, "kernels": kernels, "clocks": clk.summary(),
            "cpu_baseline": cpu, **extra}
    print(json.dumps(line), flush=True)


def time_steps(torch, fn, k):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(k):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def cpu_baseline(w, budget_s=15.0):
    o, st = w.oracle_setup()
    n, t0 = 0, time.perf_counter()
    while True:
        w.oracle_step(o, st)
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= 20:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def blas_threads():
    """Threads of the BLAS numpy uses: threadpoolctl when installed, else the
    OpenBLAS library numpy loaded, asked directly through its C API."""
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        pass
    try:
        import ctypes
        np.dot(np.ones((2, 2)), np.ones((2, 2)))   # the BLAS is loaded by now
        libs = set()
        with open("/proc/self/maps") as f:
            for line in f:
                path = line.split()[-1]
                if "openblas" in path.lower() and ".so" in path:
                    libs.add(path)
        for path in sorted(libs):
            lib = ctypes.CDLL(path)
            for fn in ("openblas_get_num_threads64_", "openblas_get_num_threads", "scipy_openblas_get_num_threads64_",
                       "scipy_openblas_get_num_threads"):
                if hasattr(lib, fn):
                    return int(getattr(lib, fn)())
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- arms

def step_config(n_gpus):
    """The default workload's config, the same on both arms."""
    return {"workload": "flashmap4b_step: append 17 rows at 1024 + 16-slot draft at 1041 (L=1042), Q8_0 vocab 151936",
            "global_batch": 16 * n_gpus, "seq_len": 1042, "parallelism": "replicas" if n_gpus > 1 else "single",
            "l2": "inputs > L2 (1.35 GB/step)"}


def run_reference(args):
    ws, rank, _ = dist()
    if rank != 0:
        return
    import torch  # noqa: F401
    from types import SimpleNamespace
    w = SimpleNamespace()
    import fm_synth as S
    from oracle import FlashMap
    cfg = S.flashmap_4b_config()
    wt = S.gen_weights(cfg, 1002)
    mod = S.gen_modulation(cfg, 1002)
    fr = S.streams(1002)["features"]
    ctx = S.gen_features(fr, 1024, cfg.feat_dim)
    f17 = S.gen_features(fr, 17, cfg.feat_dim)
    anchor = S.gen_anchor(S.streams(1002)["tokens"], cfg.vocab)
    o = FlashMap(cfg, {n: t.data for n, t in wt.items()}, mod, True)
    st = o.new_state()
    o.context_append(st, ctx, 0)
    for _ in range(args.warmup):
        o.context_append(st, f17, 1024)
        o.draft(st, anchor, 1041)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.context_append(st, f17, 1024)
        o.draft(st, anchor, 1041)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(args.gpus),
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} full steps after {args.warmup} warm-up steps",
                             "blas_threads": blas_threads()},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    ws, rank, local = dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as d
        d.init_process_group("nccl", device_id=torch.device("cuda", local))
    from block_speculative_decoding_fm_gb300 import build
    build.build()
    import block_speculative_decoding_fm_gb300 as fm
    hbm, bf16, bf16s, peak_src = peaks()

    w = FlashMapStep(torch)
    for _ in range(max(3, args.warmup)):
        w.step()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    w.launches = 0
    with Clocks(local) as clk:
        ms = time_steps(torch, w.step, args.steps)
    launches = w.launches
    ms = barrier_max(ws, ms)
    steps_s = whole_job_rate(args.steps, ws, ms)
    hbm_gbs = w.bytes_per_step * steps_s / ws / 1e9

    # end to end through the C ABI with host buffers (H2D of the feature rows,
    # D2H of the drafted tokens inside the timed region)
    e2e = None
    if not args.no_e2e:
        for _ in range(3):
            w.step_e2e()
        ms_e2e = barrier_max(ws, time_steps(torch, w.step_e2e, args.steps))
        e2e = {"value": whole_job_rate(args.steps, ws, ms_e2e), "unit": "steps/s", "h2d_bytes_per_step": w.e2e_h2d,
               "d2h_bytes_per_step": w.e2e_d2h}

    # per-kernel device time (events around every launch; a separate pass)
    roofline, kernels = None, None
    if not args.no_kprof:
        fm.fm_set_debug(w.h, fm.FM_DEBUG_PROFILE)
        for _ in range(20):
            w.step()
        prof = fm.fm_profile_read(w.h)
        fm.fm_set_debug(w.h, 0)
        top = max(prof.items(), key=lambda kv: kv[1][1])
        name, (nl, tms, tb) = top
        per_launch_ms = tms / nl
        achieved = (tb / nl) / (per_launch_ms / 1000) / 1e9
        kernels = {k: {"launches": v[0] // 20, "ms_per_step": v[1] / 20,
                       "gbs": (v[2] / v[0]) / ((v[1] / v[0]) / 1000) / 1e9} for k, v in sorted(prof.items())}
        roofline = {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "traffic": ncu_traffic(name), "peak_source": f"{peak_src} burst copy",
                    "bytes_per_launch": tb / nl, "ms_per_launch": per_launch_ms}

    extra = {}
    if not args.no_prefill and rank == 0:
        pf = PrefillStep(torch)
        pf.step()
        torch.cuda.synchronize()
        pms = time_steps(torch, pf.step, 10) / 10
        extra["prefill_rows_per_s"] = pf.rows / (pms / 1000)
        extra["prefill_reps"] = 10
        extra["prefill_tflops"] = pf.flops / (pms / 1000) / 1e12
        fm.fm_destroy(pf.h)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n, dt = cpu_baseline(w)
        cpu = {"value": v, "unit": "steps/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{n} full append+draft steps of the same workload in {dt:.1f} s",
               "blas_threads": blas_threads()}

    if rank == 0:
        line = {"metric": METRIC, "value": steps_s, "unit": "steps/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "dtype_note": "bf16 / Q8_0 weights on bf16/f16 tensor cores with split (hi + lo) activations, "
                              "f32 accumulate", "data": "synthetic",
                "config": step_config(ws),
                "achieved_hbm_gbs": hbm_gbs, "bytes_per_step": w.bytes_per_step,
                "e2e": e2e, "gpu_launches": launches, "roofline": roofline, "kernels": kernels,
                "clocks": clk.summary(), "cpu_baseline": cpu, **extra}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    global WORKLOAD
    args = parse()
    WORKLOAD = args.workload
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "flashmap4b":
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
