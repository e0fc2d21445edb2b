"""Python binding of libfm.so (include/fm.h): argument marshalling only.

Every function below has the name of the C entry point it calls and does
nothing but convert arguments (numpy / torch tensors, streams) and turn a
non-zero status into an ``FmError``.  All compute runs in the library's CUDA
kernels; there is no CPU fallback: if the library is missing or cannot load,
``load_library`` raises.  PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Iterable, Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfm.so")

# status codes (fm_status)
FM_OK, FM_ERR_INVALID_ARG, FM_ERR_UNSUPPORTED, FM_ERR_OOM, FM_ERR_CONTEXT_FULL, FM_ERR_STATE, FM_ERR_CUDA, \
    FM_ERR_TIMEOUT = range(8)
FM_VARIANT_FLASHMAP, FM_VARIANT_DFLASH = 0, 1
FM_LM_BF16, FM_LM_Q8_0 = 0, 1
FM_DTYPE_BF16, FM_DTYPE_Q8_0, FM_DTYPE_F32 = 0, 1, 2
FM_DEBUG_HIDDEN, FM_DEBUG_HEAD_OUT, FM_DEBUG_LOGITS, FM_DEBUG_CACHE_K, FM_DEBUG_CACHE_V, FM_DEBUG_H0, \
    FM_DEBUG_STEP_TRACE = range(7)
FM_DEBUG_KEEP_HIDDEN = 1
FM_DEBUG_PROFILE = 2
FM_DEBUG_TRACE = 4

EXPORTS = ["fm_create", "fm_time_conditioning", "fm_context_append", "fm_context_append_batched", "fm_draft",
           "fm_context_append_host", "fm_context_append_batched_host", "fm_draft_host", "fm_draft_pruned",
           "fm_accept", "fm_accept_batched", "fm_lm_head_argmax_noalloc", "fm_synchronize",
           "fm_selftest_wait_timeout", "fm_debug_copy", "fm_set_debug", "fm_get_length", "fm_memory_bytes",
           "fm_last_launch_count", "fm_profile_read", "fm_status_str", "fm_last_error", "fm_destroy",
           "fm_policy_init", "fm_policy_next", "fm_policy_after_round", "fm_policy_after_plain",
           "fm_mtp_create", "fm_mtp_forward", "fm_mtp_draft", "fm_mtp_cache", "fm_mtp_last_launch_count",
           "fm_mtp_last_error", "fm_mtp_destroy"]


class FmConfig(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("dim", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("ff_dim", ctypes.c_int32),
                ("block", ctypes.c_int32), ("target_dim", ctypes.c_int32), ("n_taps", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("lm_format", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
                ("max_seqs", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("ln_eps", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("qk_eps", ctypes.c_float)]


class FmTensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("data", ctypes.c_void_p), ("nbytes", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("on_device", ctypes.c_int32)]


class FmKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("ms", ctypes.c_float),
                ("bytes", ctypes.c_double)]


class FmVerifyPolicy(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int32), ("verify", ctypes.c_int32), ("fallback", ctypes.c_int32),
                ("probe_every", ctypes.c_int32), ("ema", ctypes.c_double), ("ema_tokens", ctypes.c_double),
                ("round_ms", ctypes.c_double), ("step_ms", ctypes.c_double), ("plain_left", ctypes.c_int32),
                ("rounds", ctypes.c_int32), ("catch_up", ctypes.c_int32), ("pad", ctypes.c_int32)]


FM_ACT_ROUND, FM_ACT_PLAIN, FM_ACT_PLAIN_LIMIT = 0, 1, 2


class FmMtpConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("rot_dims", ctypes.c_int32),
                ("theta", ctypes.c_float), ("eps", ctypes.c_float), ("vocab", ctypes.c_int32),
                ("kv_cap", ctypes.c_int32), ("max_rows", ctypes.c_int32)]


class FmError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfm.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run block_speculative_decoding_fm_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "fm_create": (I32, [ctypes.POINTER(FmConfig), ctypes.POINTER(FmTensor), I32, P, P, ctypes.POINTER(P)]),
        "fm_time_conditioning": (I32, [ctypes.POINTER(FmConfig), ctypes.POINTER(FmTensor), I32, I32, I32,
                                       ctypes.c_float, ctypes.c_float, ctypes.c_float, P, P]),
        "fm_context_append": (I32, [P, I32, P, I32, I32, P]),
        "fm_context_append_batched": (I32, [P, I32, P, P, P, P, P]),
        "fm_draft": (I32, [P, I32, P, P, P, P, P]),
        "fm_context_append_host": (I32, [P, I32, P, I32, I32, P]),
        "fm_context_append_batched_host": (I32, [P, I32, P, P, P, P, P]),
        "fm_draft_host": (I32, [P, I32, P, P, P, P, P]),
        "fm_draft_pruned": (I32, [P, I32, I32, I32, P, ctypes.c_float, P, P, P, P]),
        "fm_accept": (I32, [P, P, I32, P, P]),
        "fm_accept_batched": (I32, [P, I32, P, P, P, P, P, P]),
        "fm_lm_head_argmax_noalloc": (I32, [P, P, I32, P, P]),
        "fm_synchronize": (I32, [P, P]),
        "fm_selftest_wait_timeout": (I32, [P, I32, P]),
        "fm_debug_copy": (I32, [P, I32, I32, I32, I64, P, I64, P]),
        "fm_set_debug": (I32, [P, I32]),
        "fm_get_length": (I32, [P, I32, ctypes.POINTER(I32)]),
        "fm_memory_bytes": (I32, [P, ctypes.POINTER(I64)]),
        "fm_last_launch_count": (I32, [P, ctypes.POINTER(I32)]),
        "fm_profile_read": (I32, [P, ctypes.POINTER(FmKernelTime), I32, ctypes.POINTER(I32)]),
        "fm_status_str": (ctypes.c_char_p, [I32]),
        "fm_last_error": (ctypes.c_char_p, [P]),
        "fm_destroy": (None, [P]),
        "fm_policy_init": (I32, [ctypes.POINTER(FmVerifyPolicy), I32, I32, I32, I32]),
        "fm_policy_next": (I32, [ctypes.POINTER(FmVerifyPolicy), I32, I32, ctypes.POINTER(I32), ctypes.POINTER(I32)]),
        "fm_policy_after_round": (I32, [ctypes.POINTER(FmVerifyPolicy), I32, ctypes.c_double]),
        "fm_policy_after_plain": (I32, [ctypes.POINTER(FmVerifyPolicy), ctypes.c_double, I32]),
        "fm_mtp_create": (I32, [ctypes.POINTER(FmMtpConfig), ctypes.POINTER(FmTensor), I32, P, ctypes.POINTER(P)]),
        "fm_mtp_forward": (I32, [P, I32, P, P, I32, I32, P, P, P]),
        "fm_mtp_draft": (I32, [P, I32, P, P, I32, I32, I32, P, P]),
        "fm_mtp_cache": (I32, [P, I32, I32, P, P]),
        "fm_mtp_last_launch_count": (I32, [P, ctypes.POINTER(I32)]),
        "fm_mtp_last_error": (ctypes.c_char_p, [P]),
        "fm_mtp_destroy": (None, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, handle=None):
    if status != FM_OK:
        lib = load_library()
        msg = lib.fm_last_error(handle).decode() if handle is not None else lib.fm_last_error(None).decode()
        raise FmError(status, f"{lib.fm_status_str(status).decode()}: {msg}")


def make_config(cfg) -> FmConfig:
    """An FmConfig from any object with the fm_config fields."""
    return FmConfig(cfg.variant, cfg.dim, cfg.n_heads, cfg.head_dim, cfg.n_layers, cfg.ff_dim, cfg.block,
                    cfg.target_dim, cfg.n_taps, cfg.vocab, cfg.lm_format, cfg.max_ctx, cfg.max_seqs,
                    cfg.rope_theta, cfg.ln_eps, cfg.rms_eps, cfg.qk_eps)


def _tensor_array(weights):
    items = list(weights)
    keep = []
    arr = (FmTensor * max(1, len(items)))()
    for i, (name, data, dtype) in enumerate(items):
        on_dev = 0
        if isinstance(data, np.ndarray):
            data = np.ascontiguousarray(data)
            nbytes = data.nbytes
        else:
            on_dev = 1 if data.is_cuda else 0
            nbytes = data.numel() * data.element_size()
        keep.append(data)
        bname = name.encode()
        keep.append(bname)
        arr[i] = FmTensor(bname, _ptr(data), nbytes, dtype, on_dev)
    return arr, len(items), keep


def fm_time_conditioning(cfg, weights: Iterable[Tuple[str, object, int]], time_dim: int, cond_dim: int,
                         time_scale: float, s: float, t: float, table, stream=None) -> None:
    """The adaLN table of the jump s -> t into ``table`` (a CUDA float32
    tensor of (3 n_layers + 1) * 3 * dim values)."""
    lib = load_library()
    arr, n, keep = _tensor_array(weights)
    c = make_config(cfg)
    _check(lib.fm_time_conditioning(ctypes.byref(c), arr, n, time_dim, cond_dim, time_scale, s, t, _ptr(table),
                                    _stream(stream)))


def fm_create(cfg, weights: Iterable[Tuple[str, object, int]], modulation=None, stream=None) -> ctypes.c_void_p:
    """weights: (name, array, FM_DTYPE_*) triples; arrays are host numpy
    arrays or CUDA tensors (their raw bytes are passed).  modulation: a host
    array or a CUDA float32 tensor."""
    lib = load_library()
    arr, n_items, keep = _tensor_array(weights)
    items = range(n_items)
    mod = None
    if modulation is not None:
        mod = modulation if hasattr(modulation, "data_ptr") else np.ascontiguousarray(modulation, dtype=np.float32)
        keep.append(mod)
    c = make_config(cfg)
    h = ctypes.c_void_p()
    _check(lib.fm_create(ctypes.byref(c), arr, len(items), _ptr(mod), _stream(stream), ctypes.byref(h)))
    h._fm_target_dim = int(cfg.target_dim)
    h._fm_block = int(cfg.block)
    h._fm_feat = int(cfg.n_taps) * int(cfg.target_dim)
    return h


def fm_context_append(h, seq: int, feats, n_rows: int, start_pos: int, stream=None) -> None:
    lib = load_library()
    _check(lib.fm_context_append(h, seq, _ptr(feats), n_rows, start_pos, _stream(stream)), h)


def fm_context_append_batched(h, seq_ids: Sequence[int], feats, n_rows: Sequence[int], starts: Sequence[int],
                              stream=None) -> None:
    lib = load_library()
    n = len(seq_ids)
    ids = np.ascontiguousarray(seq_ids, np.int32)
    nr = np.ascontiguousarray(n_rows, np.int32)
    st = np.ascontiguousarray(starts, np.int32)
    _check(lib.fm_context_append_batched(h, n, _ptr(ids), _ptr(feats), _ptr(nr), _ptr(st), _stream(stream)), h)


def fm_draft(h, seq_ids: Sequence[int], anchors: Sequence[int], pos: Sequence[int], tokens, stream=None) -> None:
    """tokens: a CUDA int32 tensor [n_seqs, block] that receives the drafts."""
    lib = load_library()
    ids = np.ascontiguousarray(seq_ids, np.int32)
    an = np.ascontiguousarray(anchors, np.int32)
    ps = np.ascontiguousarray(pos, np.int32)
    _check(lib.fm_draft(h, len(ids), _ptr(ids), _ptr(an), _ptr(ps), _ptr(tokens), _stream(stream)), h)


def _host_buffer(x, dtype, what: str, need: int):
    """A host buffer for the host-buffer calls: a C-contiguous numpy array or
    CPU tensor of dtype with at least need elements (pinned memory keeps the
    copy asynchronous)."""
    if isinstance(x, np.ndarray):
        ok, size = x.dtype == dtype and x.flags["C_CONTIGUOUS"], x.size
    else:
        ok = not getattr(x, "is_cuda", True) and x.is_contiguous() and str(x.dtype) == "torch." + np.dtype(dtype).name
        size = x.numel() if ok else 0
    if not ok:
        raise ValueError(f"{what} must be a contiguous {np.dtype(dtype).name} host array or CPU tensor")
    if size < need:
        raise ValueError(f"{what} holds {size} values, fewer than the call's {need}")
    return x


def fm_context_append_host(h, seq: int, feats, n_rows: int, start_pos: int, stream=None) -> None:
    """fm_context_append with the rows in host memory (copied on the stream)."""
    lib = load_library()
    f = None if n_rows <= 0 else _host_buffer(feats, np.float32, "feature rows", n_rows * h._fm_feat)
    _check(lib.fm_context_append_host(h, seq, _ptr(f), n_rows, start_pos, _stream(stream)), h)


def fm_context_append_batched_host(h, seq_ids: Sequence[int], feats, n_rows: Sequence[int], starts: Sequence[int],
                                   stream=None) -> None:
    lib = load_library()
    ids = np.ascontiguousarray(seq_ids, np.int32)
    nr = np.ascontiguousarray(n_rows, np.int32)
    st = np.ascontiguousarray(starts, np.int32)
    total = int(np.maximum(nr, 0).sum())
    f = None if total == 0 else _host_buffer(feats, np.float32, "feature rows", total * h._fm_feat)
    _check(lib.fm_context_append_batched_host(h, len(ids), _ptr(ids), _ptr(f), _ptr(nr), _ptr(st),
                                              _stream(stream)), h)


def fm_draft_host(h, seq_ids: Sequence[int], anchors: Sequence[int], pos: Sequence[int], tokens, stream=None) -> None:
    """tokens: host int32 [n_seqs, block] (numpy array or CPU tensor, pinned for an
    asynchronous copy); complete once the stream has passed the call."""
    lib = load_library()
    ids = np.ascontiguousarray(seq_ids, np.int32)
    an = np.ascontiguousarray(anchors, np.int32)
    ps = np.ascontiguousarray(pos, np.int32)
    _host_buffer(tokens, np.int32, "tokens", len(ids) * h._fm_block)
    _check(lib.fm_draft_host(h, len(ids), _ptr(ids), _ptr(an), _ptr(ps), _ptr(tokens), _stream(stream)), h)


def fm_draft_pruned(h, seq: int, anchor: int, pos: int, tokens, conf=None, length=None, thresholds=None,
                    min_conf: Optional[float] = None, stream=None) -> None:
    """The DFlash draft through the sequential head with confidence pruning.
    tokens: a CUDA int32 tensor [block]; conf: a CUDA float32 tensor [block] or
    None; length: a CUDA int32 tensor [1] or None.  thresholds: per-position
    thresholds (a sequence of block floats, NaN for none) or None, in which
    case min_conf (None: no pruning) applies to every position."""
    lib = load_library()
    thr = None if thresholds is None else np.ascontiguousarray(thresholds, np.float32)
    mc = float("nan") if min_conf is None else float(min_conf)
    _check(lib.fm_draft_pruned(h, seq, anchor, pos, _ptr(thr), mc, _ptr(tokens), _ptr(conf), _ptr(length),
                               _stream(stream)), h)


def fm_accept(draft: Sequence[int], target: Sequence[int], k: int) -> Tuple[int, int]:
    lib = load_library()
    d = np.ascontiguousarray(draft, np.int32)
    t = np.ascontiguousarray(target, np.int32)
    acc, bonus = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.fm_accept(_ptr(d), _ptr(t), k, ctypes.byref(acc), ctypes.byref(bonus)))
    return acc.value, bonus.value


def fm_accept_batched(h, draft, target, k, n_accepted, bonus, stream=None) -> None:
    lib = load_library()
    _check(lib.fm_accept_batched(h, draft.shape[0], _ptr(draft), _ptr(target), _ptr(k), _ptr(n_accepted),
                                 _ptr(bonus), _stream(stream)), h)


def fm_lm_head_argmax_noalloc(h, y, tokens, stream=None) -> None:
    """The fused lm_head + argmax on caller rows, for callers that must not
    allocate device memory while they run (the library keeps its scratch in
    static device memory).  y: a CUDA float32 tensor [n_rows, target_dim]
    (n_rows <= 16); tokens: a CUDA int32 tensor [n_rows] that receives the
    argmax over the token table.  The first call on a device does a one-time
    set-up, so make it before any stream capture; overlapping calls race."""
    import torch
    if not (isinstance(y, torch.Tensor) and isinstance(tokens, torch.Tensor)):
        raise ValueError("y and tokens must be torch tensors")
    if not (y.is_cuda and tokens.is_cuda):
        raise ValueError("y and tokens must be CUDA tensors")
    if y.dtype != torch.float32 or tokens.dtype != torch.int32:
        raise ValueError("y must be float32 and tokens int32")
    if y.dim() != 2 or not y.is_contiguous() or not tokens.is_contiguous():
        raise ValueError("y must be a contiguous [n_rows, target_dim] tensor and tokens contiguous")
    width = getattr(h, "_fm_target_dim", None)
    if width is not None and y.shape[1] != width:
        raise ValueError(f"y has {y.shape[1]} columns, the drafter's target_dim is {width}")
    if tokens.numel() < y.shape[0]:
        raise ValueError("tokens holds fewer entries than y has rows")
    _check(load_library().fm_lm_head_argmax_noalloc(h, _ptr(y), y.shape[0], _ptr(tokens), _stream(stream)), h)


def fm_synchronize(h, stream=None) -> None:
    """Wait for the stream; raise FmError(FM_ERR_TIMEOUT) if a device-side
    bounded wait gave up since the last check."""
    _check(load_library().fm_synchronize(h, _stream(stream)), h)


def fm_selftest_wait_timeout(h, budget_us: int, stream=None) -> None:
    """Launch a wait that cannot complete, bounded by budget_us (the failure
    path of the bounded waits); the next fm_synchronize reports it."""
    _check(load_library().fm_selftest_wait_timeout(h, budget_us, _stream(stream)), h)


def fm_debug_copy(h, what: int, seq: int, index: int, out: np.ndarray, offset: int = 0, stream=None) -> np.ndarray:
    lib = load_library()
    _check(lib.fm_debug_copy(h, what, seq, index, offset, _ptr(out), out.nbytes, _stream(stream)), h)
    return out


def fm_set_debug(h, flags: int) -> None:
    _check(load_library().fm_set_debug(h, flags), h)


def fm_get_length(h, seq: int) -> int:
    v = ctypes.c_int32()
    _check(load_library().fm_get_length(h, seq, ctypes.byref(v)), h)
    return v.value


def fm_memory_bytes(h) -> int:
    v = ctypes.c_int64()
    _check(load_library().fm_memory_bytes(h, ctypes.byref(v)), h)
    return v.value


def fm_last_launch_count(h) -> int:
    v = ctypes.c_int32()
    _check(load_library().fm_last_launch_count(h, ctypes.byref(v)), h)
    return v.value


def fm_profile_read(h):
    """{kernel name: (launches, total ms, total algorithmic bytes)} since the last read."""
    lib = load_library()
    buf = (FmKernelTime * 64)()
    n = ctypes.c_int32()
    _check(lib.fm_profile_read(h, buf, 64, ctypes.byref(n)), h)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms, buf[i].bytes) for i in range(min(n.value, 64))}


def fm_destroy(h) -> None:
    if h is not None:
        load_library().fm_destroy(h)


def weight_items(tensors: Dict[str, object]):
    """(name, array, dtype) triples from name -> object with .data / .dtype."""
    return [(n, t.data, t.dtype) for n, t in tensors.items()]


def _mtp_check(status: int, m=None):
    if status != FM_OK:
        lib = load_library()
        raise FmError(status, f"{lib.fm_status_str(status).decode()}: {lib.fm_mtp_last_error(m).decode()}")


def fm_mtp_create(cfg, weights: Iterable[Tuple[str, object, int]], stream=None) -> ctypes.c_void_p:
    """The MTP draft head.  cfg: any object with the fm_mtp_config fields;
    weights: (name, array, FM_DTYPE_*) triples (host arrays or CUDA tensors)."""
    lib = load_library()
    arr, n_items, keep = _tensor_array(weights)
    c = FmMtpConfig(cfg.hidden, cfg.inter, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rot_dims, cfg.theta, cfg.eps,
                    cfg.vocab, cfg.kv_cap, cfg.max_rows)
    m = ctypes.c_void_p()
    _mtp_check(lib.fm_mtp_create(ctypes.byref(c), arr, n_items, _stream(stream), ctypes.byref(m)))
    return m


def fm_mtp_forward(m, tokens, hn, pos0: int, kv_lo: int, hout=None, drafts=None, stream=None) -> None:
    """One pass over len(tokens) rows.  tokens: CUDA int32 [M]; hn: CUDA float32
    [M, H]; hout: CUDA float32 [M, H] or None; drafts: CUDA int32 [M] or None."""
    _mtp_check(load_library().fm_mtp_forward(m, int(tokens.shape[0]), _ptr(tokens), _ptr(hn), pos0, kv_lo, _ptr(hout),
                                             _ptr(drafts), _stream(stream)), m)


def fm_mtp_draft(m, tokens, hn, pos0: int, kv_lo: int, depth: int, drafts, stream=None) -> None:
    """A pass over the pending rows then depth - 1 chained single-row passes;
    drafts: CUDA int32 [depth]."""
    _mtp_check(load_library().fm_mtp_draft(m, int(tokens.shape[0]), _ptr(tokens), _ptr(hn), pos0, kv_lo, depth,
                                           _ptr(drafts), _stream(stream)), m)


def fm_mtp_cache(m, which: int, rows: int, out: np.ndarray, stream=None) -> np.ndarray:
    """Copy K (0) or V (1) cache rows [0, rows) into a host float32 array."""
    _mtp_check(load_library().fm_mtp_cache(m, which, rows, _ptr(out), _stream(stream)), m)
    return out


def fm_mtp_last_launch_count(m) -> int:
    n = ctypes.c_int32()
    _mtp_check(load_library().fm_mtp_last_launch_count(m, ctypes.byref(n)), m)
    return n.value


def fm_mtp_destroy(m) -> None:
    if m is not None:
        load_library().fm_mtp_destroy(m)


def fm_policy_init(block: int, verify: int = 0, fallback: bool = True, probe_every: int = 16) -> FmVerifyPolicy:
    p = FmVerifyPolicy()
    _check(load_library().fm_policy_init(ctypes.byref(p), block, verify, 1 if fallback else 0, probe_every))
    return p


def fm_policy_next(p: FmVerifyPolicy, position: int, max_ctx: int) -> Tuple[int, int]:
    """(action, k): FM_ACT_ROUND with the verify length, or a plain step."""
    a, k = ctypes.c_int32(), ctypes.c_int32()
    _check(load_library().fm_policy_next(ctypes.byref(p), position, max_ctx, ctypes.byref(a), ctypes.byref(k)))
    return a.value, k.value


def fm_policy_after_round(p: FmVerifyPolicy, accepted: int, ms: float) -> None:
    _check(load_library().fm_policy_after_round(ctypes.byref(p), accepted, ms))


def fm_policy_after_plain(p: FmVerifyPolicy, ms: float, rows_handed: bool) -> None:
    _check(load_library().fm_policy_after_plain(ctypes.byref(p), ms, 1 if rows_handed else 0))
