"""CONF-KV decode-step cache manager for GB300: thin Python binding.

This module only marshals arguments to the C ABI declared in
``include/confkv.h`` (``libconfkv.so``, built in-tree by ``build.py``).  Every
step of the path runs in the library's CUDA kernels; if the library is
missing, importing the binding's entry points raises -- there is no CPU
fallback.

Method: CONF-KV (confidence-aware KV cache eviction with mixed-precision
storage), gist.science summaries of paper 2605.24786, "Technische
Samenvatting".
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libconfkv.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_CUDA = -2
ERR_OOM = -3
ERR_CAPACITY = -4
ERR_NONFINITE_LOGITS = -5
ERR_STATE = -6
ERR_DEVICE = -7
POLICY_CONFKV, POLICY_WINDOW, POLICY_H2O, POLICY_RANDOM = 0, 1, 2, 3
FLAG_NONFINITE = 1
FLAG_CAPACITY = 2
FLAG_TIMEOUT = 4

# every symbol declared in include/confkv.h
EXPORTS = ("confkv_create", "confkv_prefill", "confkv_step", "confkv_step_host",
           "confkv_stats", "confkv_read_cache", "confkv_profile_enable",
           "confkv_profile_read", "confkv_last_error", "confkv_free",
           "confkv_confidence_noalloc", "confkv_step_begin", "confkv_step_layer",
           "confkv_attention_path", "confkv_selftest_bounded_wait",
           "confkv_read_channel_exponents")


def selftest_bounded_wait(device=0, timeout_us=1000):
    """Runs confkv_selftest_bounded_wait; returns (gave_up, waited_us)."""
    L = load_library()
    g = ctypes.c_int()
    w = ctypes.c_double()
    rc = L.confkv_selftest_bounded_wait(int(device), int(timeout_us), ctypes.byref(g), ctypes.byref(w))
    if rc != OK:
        raise ConfKVError(rc, "bounded-wait self-test")
    return bool(g.value), w.value


class ConfKVError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"confkv error {code}: {msg}")
        self.code = code


class Opts(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("vocab", ctypes.c_int),
                ("max_context", ctypes.c_int), ("pyramid_min", ctypes.c_float),
                ("device", ctypes.c_int), ("attn_splits", ctypes.c_int),
                ("attn_kernel", ctypes.c_int), ("attn_tma", ctypes.c_int),
                ("policy", ctypes.c_int), ("int8_channel", ctypes.c_int), ("seed", ctypes.c_uint64)]


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("position", ctypes.c_int64),
                ("error_flags", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("tokens_evicted", ctypes.c_int64), ("tokens_quantized", ctypes.c_int64),
                ("tokens_moved", ctypes.c_int64), ("cache_tokens", ctypes.c_int64),
                ("attn_kv_bytes", ctypes.c_int64), ("logits_bytes", ctypes.c_int64),
                ("budget_high_steps", ctypes.c_int64), ("cache_bytes", ctypes.c_double),
                ("kernel_launches", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class Profile(ctypes.Structure):
    _fields_ = [("n_kernels", ctypes.c_int32), ("launches", ctypes.c_int32 * 8),
                ("total_ms", ctypes.c_double * 8), ("names", ctypes.c_char_p * 8)]


_lib = None


def load_library(path=LIB_PATH):
    """Load libconfkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "confidence_gated_kv_logits_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.confkv_create.restype = ci
    L.confkv_create.argtypes = [ci, ci, ci, ci, ci, ci, cf, ci, ci, cf,
                                ctypes.POINTER(Opts), ctypes.POINTER(vp)]
    L.confkv_prefill.restype = ci
    L.confkv_prefill.argtypes = [vp, vp, vp, ci, vp, vp]
    L.confkv_step.restype = ci
    L.confkv_step.argtypes = [vp] * 11
    L.confkv_step_begin.restype = ci
    L.confkv_step_begin.argtypes = [vp] * 5
    L.confkv_step_layer.restype = ci
    L.confkv_step_layer.argtypes = [vp, ci] + [vp] * 7
    L.confkv_step_host.restype = ci
    L.confkv_step_host.argtypes = [vp] * 11
    L.confkv_stats.restype = ci
    L.confkv_stats.argtypes = [vp, ctypes.POINTER(Stats)]
    L.confkv_read_cache.restype = ci
    L.confkv_read_cache.argtypes = [vp, ci, ci, ci, vp, vp] + [vp] * 9
    L.confkv_profile_enable.restype = ci
    L.confkv_profile_enable.argtypes = [vp, ci]
    L.confkv_profile_read.restype = ci
    L.confkv_profile_read.argtypes = [vp, ctypes.POINTER(Profile)]
    L.confkv_last_error.restype = ctypes.c_char_p
    L.confkv_last_error.argtypes = [vp]
    L.confkv_free.restype = None
    L.confkv_free.argtypes = [vp]
    L.confkv_selftest_bounded_wait.restype = ci
    L.confkv_selftest_bounded_wait.argtypes = [ci, ci, ctypes.POINTER(ci), ctypes.POINTER(ctypes.c_double)]
    L.confkv_attention_path.restype = ci
    L.confkv_attention_path.argtypes = [vp]
    L.confkv_read_channel_exponents.restype = ci
    L.confkv_read_channel_exponents.argtypes = [vp, ci, ci, vp, vp]
    L.confkv_confidence_noalloc.restype = ci
    L.confkv_confidence_noalloc.argtypes = [vp, ci, ci, cf, ci, ci, vp, vp, vp, vp]
    _lib = L
    return L


def _dptr(t, dtype, numel, name, device):
    """Device pointer of a contiguous torch tensor (argument checks only)."""
    if t is None:
        return None
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != dtype or not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{name}: want contiguous {dtype} with {numel} elements, got "
                         f"{t.dtype} {tuple(t.shape)}")
    return t.data_ptr()


def _hptr(a, np_dtype, numel, name):
    """Address of a C-contiguous numpy array (argument checks only)."""
    if a is None:
        return None
    if a.dtype != np_dtype or not a.flags.c_contiguous or a.size != numel:
        raise ValueError(f"{name}: want C-contiguous {np_dtype} with {numel} elements")
    return a.ctypes.data


class ConfKV:
    """One CONF-KV cache manager (all layers x sequences of a batch)."""

    def __init__(self, layers, heads, kv_heads, head_dim, N_low, N_high, tau, P, W,
                 ema_decay, *, batch=1, vocab, max_context=0, pyramid_min=1.0,
                 device=None, attn_splits=0, attn_kernel=0, attn_tma=0, policy=0, seed=0,
                 int8_channel=0):
        import torch
        self._L = load_library()
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.device = dev
        opts = Opts(batch, vocab, max_context, pyramid_min, dev.index, attn_splits, attn_kernel,
                    attn_tma, policy, int8_channel, seed)
        self.policy = policy
        h = ctypes.c_void_p()
        rc = self._L.confkv_create(layers, heads, kv_heads, head_dim, N_low, N_high, tau, P,
                                   W, ema_decay, ctypes.byref(opts), ctypes.byref(h))
        if rc != OK:
            raise ConfKVError(rc, "confkv_create failed")
        self._h = h
        self.L, self.B, self.Hq, self.Hkv, self.d, self.V = (layers, batch, heads, kv_heads,
                                                             head_dim, vocab)
        self.N_low, self.N_high, self.P, self.W = N_low, N_high, P, W
        self.Ncap = max(N_low, N_high)

    @classmethod
    def for_workload(cls, w, **kw):
        kw.setdefault("int8_channel", getattr(w, "int8_channel", 0))
        return cls(w.L, w.Hq, w.Hkv, w.d, w.N_low, w.N_high, w.tau, w.P, w.W, w.beta,
                   batch=w.B, vocab=w.V, max_context=w.prefill, pyramid_min=w.pyramid_min,
                   **kw)

    def close(self):
        if getattr(self, "_h", None):
            self._L.confkv_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != OK:
            raise ConfKVError(rc, self._L.confkv_last_error(self._h).decode())

    @staticmethod
    def _stream(stream):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        return s.cuda_stream

    def prefill(self, k, v, T, q_last=None, stream=None):
        import torch
        L, B, H, d = self.L, self.B, self.Hkv, self.d
        kp = _dptr(k, torch.float16, L * B * H * T * d, "k", self.device) if T else None
        vp = _dptr(v, torch.float16, L * B * H * T * d, "v", self.device) if T else None
        qp = _dptr(q_last, torch.float16, L * B * self.Hq * d, "q_last", self.device)
        self._check(self._L.confkv_prefill(self._h, kp, vp, T, qp, self._stream(stream)))

    def step(self, logits, q, k_new, v_new, out, kept_pos=None, kept_count=None,
             conf=None, budget=None, stream=None):
        import torch
        L, B, d, dev = self.L, self.B, self.d, self.device
        args = [_dptr(logits, torch.float32, B * self.V, "logits", dev),
                _dptr(q, torch.float16, L * B * self.Hq * d, "q", dev),
                _dptr(k_new, torch.float16, L * B * self.Hkv * d, "k_new", dev),
                _dptr(v_new, torch.float16, L * B * self.Hkv * d, "v_new", dev),
                _dptr(out, torch.float32, L * B * self.Hq * d, "out", dev),
                _dptr(kept_pos, torch.int32, L * B * self.Ncap, "kept_pos", dev),
                _dptr(kept_count, torch.int32, L * B, "kept_count", dev),
                _dptr(conf, torch.float32, B, "conf", dev),
                _dptr(budget, torch.int32, B, "budget", dev)]
        self._check(self._L.confkv_step(self._h, *args, self._stream(stream)))

    def step_begin(self, logits, conf=None, budget=None, stream=None):
        import torch
        B, dev = self.B, self.device
        self._check(self._L.confkv_step_begin(
            self._h, _dptr(logits, torch.float32, B * self.V, "logits", dev),
            _dptr(conf, torch.float32, B, "conf", dev), _dptr(budget, torch.int32, B, "budget", dev),
            self._stream(stream)))

    def step_layer(self, layer, q, k_new, v_new, out, kept_pos=None, kept_count=None, stream=None):
        """One layer of a begun step; buffers hold that layer only ([B, ...])."""
        import torch
        B, d, dev = self.B, self.d, self.device
        args = [_dptr(q, torch.float16, B * self.Hq * d, "q", dev),
                _dptr(k_new, torch.float16, B * self.Hkv * d, "k_new", dev),
                _dptr(v_new, torch.float16, B * self.Hkv * d, "v_new", dev),
                _dptr(out, torch.float32, B * self.Hq * d, "out", dev),
                _dptr(kept_pos, torch.int32, B * self.Ncap, "kept_pos", dev),
                _dptr(kept_count, torch.int32, B, "kept_count", dev)]
        self._check(self._L.confkv_step_layer(self._h, layer, *args, self._stream(stream)))

    def step_host(self, logits, q, k_new, v_new, out, kept_pos=None, kept_count=None,
                  conf=None, budget=None, stream=None):
        """Host (numpy) buffers; copies happen inside the library call."""
        import numpy as np
        L, B, d = self.L, self.B, self.d
        args = [_hptr(logits, np.float32, B * self.V, "logits"),
                _hptr(q, np.float16, L * B * self.Hq * d, "q"),
                _hptr(k_new, np.float16, L * B * self.Hkv * d, "k_new"),
                _hptr(v_new, np.float16, L * B * self.Hkv * d, "v_new"),
                _hptr(out, np.float32, L * B * self.Hq * d, "out"),
                _hptr(kept_pos, np.int32, L * B * self.Ncap, "kept_pos"),
                _hptr(kept_count, np.int32, L * B, "kept_count"),
                _hptr(conf, np.float32, B, "conf"),
                _hptr(budget, np.int32, B, "budget")]
        self._check(self._L.confkv_step_host(self._h, *args, self._stream(stream)))

    ATTN_PATHS = ("cuda-core", "tensor-core cp.async", "tensor-core TMA")

    def attention_path(self):
        """Name of the attention kernel this context runs."""
        r = self._L.confkv_attention_path(self._h)
        if r < 0:
            self._check(r)
        return self.ATTN_PATHS[r]

    def stats(self, check=True):
        s = Stats()
        rc = self._L.confkv_stats(self._h, ctypes.byref(s))
        if check:
            self._check(rc)
        return s.as_dict(), rc

    def read_cache(self, l, b):
        import numpy as np
        n8 = ctypes.c_int()
        n16 = ctypes.c_int()
        self._check(self._L.confkv_read_cache(self._h, l, b, 0, ctypes.byref(n8),
                                              ctypes.byref(n16), *([None] * 9)))
        a, c = n8.value, n16.value
        H, d = self.Hkv, self.d
        r = dict(pos=np.zeros(a + c, np.int32), ema=np.zeros(a + c, np.float32),
                 k8=np.zeros((a, H, d), np.int8), v8=np.zeros((a, H, d), np.int8),
                 ks=np.zeros((a, H), np.float32), vs=np.zeros((a, H), np.float32),
                 k16=np.zeros((c, H, d), np.uint16), v16=np.zeros((c, H, d), np.uint16),
                 mass=np.zeros(a + c, np.float32))
        ptr = lambda x: x.ctypes.data_as(ctypes.c_void_p)
        self._check(self._L.confkv_read_cache(
            self._h, l, b, a + c, ctypes.byref(n8), ctypes.byref(n16),
            *[ptr(r[x]) for x in ("pos", "ema", "k8", "v8", "ks", "vs", "k16", "v16", "mass")]))
        r["n8"], r["n16"] = a, c
        return r

    def read_channel_exponents(self, l, b):
        """Channel exponents (fk, fv) of (l, b): int8 [Hkv, d] each."""
        import numpy as np
        fk = np.zeros((self.Hkv, self.d), np.int8)
        fv = np.zeros((self.Hkv, self.d), np.int8)
        self._check(self._L.confkv_read_channel_exponents(
            self._h, l, b, fk.ctypes.data_as(ctypes.c_void_p), fv.ctypes.data_as(ctypes.c_void_p)))
        return fk, fv

    KERNELS = ("confidence", "select", "append", "attention")

    def profile(self, kernels=()):
        """Time the named kernels with CUDA events (empty: off)."""
        mask = 0
        for k in kernels:
            mask |= 1 << self.KERNELS.index(k)
        self._check(self._L.confkv_profile_enable(self._h, mask))

    def profile_read(self):
        p = Profile()
        self._check(self._L.confkv_profile_read(self._h, ctypes.byref(p)))
        return {p.names[i].decode(): (p.launches[i], p.total_ms[i]) for i in range(p.n_kernels)}
