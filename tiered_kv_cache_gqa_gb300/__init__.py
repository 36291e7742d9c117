"""tkv: tiered KV-cache decode attention for one GB300 (sm_103a).

A thin ctypes binding over ``libtkv.so`` (C ABI in ``include/tkv.h``): the
functions below carry the C names and only marshal arguments (tensor data
pointers, CUDA stream handles, host buffers).  Every step of the hot path runs
in the library's CUDA kernels; there is no fallback.  If the library has not
been built, every call raises ``TkvUnavailable``.

Build with ``python -c "import tiered_kv_cache_gqa_gb300.build as b; b.build()"``.
"""

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# TKV_LIBRARY may name another build of the same library (e.g. a tuning variant).
LIB_PATH = os.environ.get("TKV_LIBRARY") or os.path.join(_HERE, "libtkv.so")

TKV_OK, TKV_EINVAL, TKV_ENOMEM, TKV_ECUDA, TKV_ECAPACITY, TKV_ETIMEOUT, TKV_ESTATE = range(7)
TKV_T1_COPY_ENGINE, TKV_T1_SM_COPY, TKV_T1_SPLIT, TKV_T1_MULTI_CE, TKV_T1_RESIDENT = range(5)
TKV_T2_HBM, TKV_T2_HOST = range(2)
TKV_HOST_AUTO, TKV_HOST_PINNED_ALLOC, TKV_HOST_HUGE_ARENA = range(3)

# Every function the C ABI exports (include/tkv.h).
EXPORTS = ("tkv_create", "tkv_destroy", "tkv_append", "tkv_prefetch", "tkv_decode_step",
           "tkv_retier", "tkv_get_scores", "tkv_set_scores", "tkv_get_tiers", "tkv_set_tiers",
           "tkv_get_row", "tkv_profile_begin", "tkv_profile_end", "tkv_sync", "tkv_get_stats",
           "tkv_status_string", "tkv_decode_dense_noalloc", "tkv_capture_begin", "tkv_capture_end",
           "tkv_replay", "tkv_measure_host_link")


class TkvUnavailable(RuntimeError):
    pass


class TkvError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, status_string(status), status))


class Config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
        ("prompt_len", ctypes.c_int32), ("num_sinks", ctypes.c_int32),
        ("recent_window", ctypes.c_int32), ("retier_interval", ctypes.c_int32),
        ("ratio_t0", ctypes.c_float), ("ratio_t1", ctypes.c_float),
        ("ratio_t2", ctypes.c_float), ("ratio_t3", ctypes.c_float),
        ("t0_capacity", ctypes.c_int32), ("t1_capacity", ctypes.c_int32),
        ("t2_capacity", ctypes.c_int32), ("t1_transport", ctypes.c_int32),
        ("device", ctypes.c_int32),
        ("compute_stream", ctypes.c_void_p), ("copy_stream", ctypes.c_void_p),
        ("t2_placement", ctypes.c_int32), ("host_alloc", ctypes.c_int32),
    ]


class Stats(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int64), ("step", ctypes.c_int64), ("retiers", ctypes.c_int64),
        ("tier_count", ctypes.c_int64 * 4), ("t1_rows_streamed", ctypes.c_int64),
        ("last_promoted", ctypes.c_int64), ("last_demoted_t1", ctypes.c_int64),
        ("last_quantised", ctypes.c_int64), ("last_evicted", ctypes.c_int64),
        ("last_t2_to_t1", ctypes.c_int64), ("h2d_bytes_t1_stream", ctypes.c_int64),
        ("h2d_bytes_delta", ctypes.c_int64), ("d2h_bytes_writeback", ctypes.c_int64),
        ("hbm_bytes_allocated", ctypes.c_int64), ("host_bytes_allocated", ctypes.c_int64),
        ("hbm_bytes_kv_resident", ctypes.c_int64), ("kv_bytes_full_cache", ctypes.c_int64),
        ("kernel_launches", ctypes.c_int64),
        ("status", ctypes.c_int32), ("attn_splits", ctypes.c_int32),
        ("h2d_bytes_t2_stream", ctypes.c_int64), ("host_huge_bytes", ctypes.c_int64),
        ("host_numa_node", ctypes.c_int32), ("cuda_error", ctypes.c_int32),
        ("cuda_error_line", ctypes.c_int32), ("pad0", ctypes.c_int32),
    ]

    def as_dict(self):
        d = {}
        for name, _ in self._fields_:
            v = getattr(self, name)
            d[name] = list(v) if name == "tier_count" else int(v)
        return d


class ProfEntry(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double), ("count", ctypes.c_int64), ("bytes", ctypes.c_double)]

    def as_dict(self):
        return {"ms": self.ms, "count": int(self.count), "bytes": self.bytes}


_lib = None


def load():
    """Loads libtkv.so (once) and declares every exported signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise TkvUnavailable("libtkv.so is not built (%s); run the build first" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int
    lib.tkv_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(vp)]
    lib.tkv_destroy.argtypes = [vp]
    lib.tkv_destroy.restype = None
    lib.tkv_append.argtypes = [vp, i32, vp, vp, i32]
    lib.tkv_prefetch.argtypes = [vp, i32]
    lib.tkv_decode_step.argtypes = [vp, i32, vp, vp]
    lib.tkv_retier.argtypes = [vp]
    lib.tkv_get_scores.argtypes = [vp, vp]
    lib.tkv_set_scores.argtypes = [vp, vp]
    lib.tkv_get_tiers.argtypes = [vp, vp]
    lib.tkv_set_tiers.argtypes = [vp, vp]
    lib.tkv_get_row.argtypes = [vp, i32, i32, i32, vp, vp, ctypes.POINTER(i32)]
    lib.tkv_profile_begin.argtypes = [vp]
    lib.tkv_profile_end.argtypes = [vp, ctypes.POINTER(ProfEntry), ctypes.POINTER(ProfEntry),
                                    ctypes.POINTER(ProfEntry), ctypes.POINTER(ProfEntry)]
    lib.tkv_decode_dense_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.tkv_capture_begin.argtypes = [vp]
    lib.tkv_capture_end.argtypes = [vp, ctypes.POINTER(i32)]
    lib.tkv_replay.argtypes = [vp]
    lib.tkv_sync.argtypes = [vp]
    dp = ctypes.POINTER(ctypes.c_double)
    lib.tkv_measure_host_link.argtypes = [i32, ctypes.c_int64, dp, dp, dp]
    lib.tkv_get_stats.argtypes = [vp, ctypes.POINTER(Stats)]
    lib.tkv_status_string.argtypes = [st]
    lib.tkv_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("tkv_destroy", "tkv_status_string"):
            getattr(lib, name).restype = st
    _lib = lib
    return lib


def status_string(s):
    return load().tkv_status_string(int(s)).decode()


def _check(rc, where):
    if rc != TKV_OK:
        raise TkvError(rc, where)


def _ptr(x):
    """Device pointer of a torch tensor, or an int address."""
    if hasattr(x, "data_ptr"):
        return ctypes.c_void_p(x.data_ptr())
    return ctypes.c_void_p(int(x))


# ------------------------------------------------------------ C-named calls
def tkv_create(cfg: Config):
    ctx = ctypes.c_void_p()
    _check(load().tkv_create(ctypes.byref(cfg), ctypes.byref(ctx)), "tkv_create")
    return ctx


def tkv_destroy(ctx):
    load().tkv_destroy(ctx)


def tkv_append(ctx, layer, k, v, n_tokens):
    return load().tkv_append(ctx, int(layer), _ptr(k), _ptr(v), int(n_tokens))


def tkv_prefetch(ctx, layer):
    return load().tkv_prefetch(ctx, int(layer))


def tkv_decode_step(ctx, layer, q, out):
    return load().tkv_decode_step(ctx, int(layer), _ptr(q), _ptr(out))


def tkv_retier(ctx):
    return load().tkv_retier(ctx)


def tkv_capture_begin(ctx):
    return load().tkv_capture_begin(ctx)


def tkv_capture_end(ctx):
    """Returns (status, replays the captured step stays valid for)."""
    n = ctypes.c_int32(0)
    rc = load().tkv_capture_end(ctx, ctypes.byref(n))
    return rc, int(n.value)


def tkv_replay(ctx):
    return load().tkv_replay(ctx)


def tkv_get_scores(ctx, dst: np.ndarray):
    assert dst.dtype == np.float32 and dst.flags["C_CONTIGUOUS"]
    return load().tkv_get_scores(ctx, dst.ctypes.data_as(ctypes.c_void_p))


def tkv_set_scores(ctx, src: np.ndarray):
    src = np.ascontiguousarray(src, dtype=np.float32)
    return load().tkv_set_scores(ctx, src.ctypes.data_as(ctypes.c_void_p))


def tkv_get_tiers(ctx, dst: np.ndarray):
    assert dst.dtype == np.uint8 and dst.flags["C_CONTIGUOUS"]
    return load().tkv_get_tiers(ctx, dst.ctypes.data_as(ctypes.c_void_p))


def tkv_set_tiers(ctx, src: np.ndarray):
    src = np.ascontiguousarray(src, dtype=np.uint8)
    return load().tkv_set_tiers(ctx, src.ctypes.data_as(ctypes.c_void_p))


def tkv_get_row(ctx, layer, seq, pos, dst: np.ndarray, scales: np.ndarray = None):
    """Returns (status, tier); dst/scales are filled in place (see include/tkv.h)."""
    t = ctypes.c_int32(-1)
    sp = scales.ctypes.data_as(ctypes.c_void_p) if scales is not None else None
    rc = load().tkv_get_row(ctx, int(layer), int(seq), int(pos), dst.ctypes.data_as(ctypes.c_void_p),
                            sp, ctypes.byref(t))
    return rc, int(t.value)


def tkv_profile_begin(ctx):
    return load().tkv_profile_begin(ctx)


def tkv_profile_end(ctx):
    """Returns (status, {"attn": ..., "combine": ..., "t1": ..., "delta": ...}) of ProfEntry dicts."""
    e = [ProfEntry(), ProfEntry(), ProfEntry(), ProfEntry()]
    rc = load().tkv_profile_end(ctx, *(ctypes.byref(x) for x in e))
    return rc, {"attn": e[0].as_dict(), "combine": e[1].as_dict(), "t1": e[2].as_dict(),
                "delta": e[3].as_dict()}


def tkv_decode_dense_noalloc(q, kv, out, s, num_layers, batch, num_q_heads, num_kv_heads,
                             head_dim, num_positions, stream=None):
    """Allocation-free decode step over a dense cache (see include/tkv.h); returns the status."""
    if stream is None:
        stream = torch_stream_handle()
    return load().tkv_decode_dense_noalloc(_ptr(q), _ptr(kv), _ptr(out), _ptr(s), int(num_layers),
                                           int(batch), int(num_q_heads), int(num_kv_heads),
                                           int(head_dim), int(num_positions), ctypes.c_void_p(stream))


def tkv_measure_host_link(device, nbytes):
    """Returns (status, {"h2d_ce_gbs", "h2d_sm_gbs", "d2h_ce_gbs"}) (see include/tkv.h)."""
    v = [ctypes.c_double(0.0) for _ in range(3)]
    rc = load().tkv_measure_host_link(int(device), int(nbytes), *(ctypes.byref(x) for x in v))
    return rc, {"h2d_ce_gbs": v[0].value, "h2d_sm_gbs": v[1].value, "d2h_ce_gbs": v[2].value}


def tkv_sync(ctx):
    return load().tkv_sync(ctx)


def tkv_get_stats(ctx):
    s = Stats()
    _check(load().tkv_get_stats(ctx, ctypes.byref(s)), "tkv_get_stats")
    return s


CUDA_STREAM_LEGACY = 1   # cudaStreamLegacy: the legacy default stream


def torch_stream_handle(stream=None):
    """cudaStream_t of a torch stream (default: the current one).  torch's default stream
    has handle 0, which the C ABI reads as "create a stream"; it is passed as the
    explicit legacy-stream handle instead, so library work is ordered with torch's."""
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    return st.cuda_stream or CUDA_STREAM_LEGACY


# --------------------------------------------------------------- wrapper
class TieredKV:
    """Owns one context; raises TkvError on any non-OK status."""

    def __init__(self, *, num_layers, num_q_heads, num_kv_heads, head_dim, batch, max_tokens,
                 prompt_len, num_sinks=4, recent_window=64, retier_interval=64,
                 ratios=(1.0, 0.0, 0.0, 0.0), t0_capacity=0, t1_capacity=0, t2_capacity=0,
                 t1_transport=TKV_T1_COPY_ENGINE, device=0, compute_stream=None, copy_stream=None,
                 t2_placement=TKV_T2_HBM, host_alloc=TKV_HOST_AUTO):
        cfg = Config()
        cfg.num_layers, cfg.num_q_heads, cfg.num_kv_heads = num_layers, num_q_heads, num_kv_heads
        cfg.head_dim, cfg.batch, cfg.max_tokens = head_dim, batch, max_tokens
        cfg.prompt_len, cfg.num_sinks, cfg.recent_window = prompt_len, num_sinks, recent_window
        cfg.retier_interval = retier_interval
        cfg.ratio_t0, cfg.ratio_t1, cfg.ratio_t2, cfg.ratio_t3 = ratios
        cfg.t0_capacity, cfg.t1_capacity, cfg.t2_capacity = t0_capacity, t1_capacity, t2_capacity
        cfg.t1_transport = t1_transport
        cfg.t2_placement = t2_placement
        cfg.host_alloc = host_alloc
        cfg.device = device
        if compute_stream is None:
            compute_stream = torch_stream_handle()
        cfg.compute_stream = compute_stream or 0
        cfg.copy_stream = copy_stream or 0
        self.cfg = cfg
        self.B, self.L, self.Hq, self.Hkv, self.d = batch, num_layers, num_q_heads, num_kv_heads, head_dim
        self.ctx = tkv_create(cfg)

    @classmethod
    def for_workload(cls, wl, **kw):
        return cls(num_layers=wl.num_layers, num_q_heads=wl.num_q_heads,
                   num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim, batch=wl.batch,
                   max_tokens=kw.pop("max_tokens", wl.max_tokens), prompt_len=wl.prompt_len,
                   num_sinks=wl.num_sinks, recent_window=wl.window, retier_interval=wl.delta,
                   ratios=kw.pop("ratios", wl.ratios), **kw)

    def close(self):
        if self.ctx is not None:
            tkv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc, where):
        if rc != TKV_OK:
            err = TkvError(rc, where)
            if rc in (TKV_ECUDA, TKV_ESTATE) and self.ctx is not None:
                st = tkv_get_stats(self.ctx)
                err.cuda_error, err.cuda_error_line = int(st.cuda_error), int(st.cuda_error_line)
                err.args = (err.args[0] + " [cudaError %d at library line %d]" % (err.cuda_error,
                                                                                   err.cuda_error_line),)
            raise err

    def append(self, layer, k, v, n_tokens=1):
        self._check(tkv_append(self.ctx, layer, k, v, n_tokens), "tkv_append")

    def prefetch(self, layer):
        self._check(tkv_prefetch(self.ctx, layer), "tkv_prefetch")

    def decode_step(self, layer, q, out):
        self._check(tkv_decode_step(self.ctx, layer, q, out), "tkv_decode_step")

    def retier(self):
        self._check(tkv_retier(self.ctx), "tkv_retier")

    def capture_begin(self):
        self._check(tkv_capture_begin(self.ctx), "tkv_capture_begin")

    def capture_end(self):
        """Ends a capture; returns how many replays the captured step stays valid for."""
        rc, n = tkv_capture_end(self.ctx)
        self._check(rc, "tkv_capture_end")
        return n

    def replay(self):
        self._check(tkv_replay(self.ctx), "tkv_replay")

    def sync(self):
        self._check(tkv_sync(self.ctx), "tkv_sync")

    def profile_begin(self):
        self._check(tkv_profile_begin(self.ctx), "tkv_profile_begin")

    def profile_end(self):
        rc, prof = tkv_profile_end(self.ctx)
        self._check(rc, "tkv_profile_end")
        return prof

    def stats(self):
        return tkv_get_stats(self.ctx).as_dict()

    def num_tokens(self):
        return int(tkv_get_stats(self.ctx).num_tokens)

    def scores(self):
        n = self.num_tokens()
        out = np.zeros((self.B, n), dtype=np.float32)
        self._check(tkv_get_scores(self.ctx, out), "tkv_get_scores")
        return out

    def set_scores(self, s):
        self._check(tkv_set_scores(self.ctx, np.asarray(s, dtype=np.float32)), "tkv_set_scores")

    def tiers(self):
        n = self.num_tokens()
        out = np.zeros((self.B, n), dtype=np.uint8)
        self._check(tkv_get_tiers(self.ctx, out), "tkv_get_tiers")
        return out

    def row(self, layer, seq, pos):
        """(tier, data, scales): bf16 bits uint16 [2][Hkv][d] for T0/T1, E4M3 codes uint8 and
        fp32 scales [2][Hkv] for T2, None for T3."""
        buf = np.zeros(2 * self.Hkv * self.d * 2, dtype=np.uint8)
        sc = np.zeros((2, self.Hkv), dtype=np.float32)
        rc, tier = tkv_get_row(self.ctx, layer, seq, pos, buf, sc)
        self._check(rc, "tkv_get_row")
        if tier in (0, 1):
            return tier, buf.view(np.uint16).reshape(2, self.Hkv, self.d), None
        if tier == 2:
            return tier, buf[: 2 * self.Hkv * self.d].reshape(2, self.Hkv, self.d), sc
        return tier, None, None

    def set_tiers(self, t):
        self._check(tkv_set_tiers(self.ctx, np.asarray(t, dtype=np.uint8)), "tkv_set_tiers")
