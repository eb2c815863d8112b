"""CPU oracle of the CONF-KV decode step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it.

The arithmetic lives in ``confkv_oracle.cpp`` (plain single-threaded C++,
fp64 except the fp32 quantiser and EMA/ranking key); this module only builds
it with g++ and marshals numpy arrays through ctypes.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "confkv_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libconfkv_oracle.so")
_lib = None


def build(force=False):
    """Compile the oracle with g++ (no fp contraction, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("L", "B", "Hq", "Hkv", "d", "V", "N_low", "N_high", "P", "W")] + [
        ("tau", ctypes.c_float), ("beta", ctypes.c_float), ("pyramid_min", ctypes.c_double),
        ("policy", ctypes.c_int), ("int8_channel", ctypes.c_int), ("seed", ctypes.c_uint64)]

POLICY_CONFKV, POLICY_WINDOW, POLICY_H2O, POLICY_RANDOM = 0, 1, 2, 3


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp = ctypes.c_void_p
        L.orc_confidence.restype = ctypes.c_double
        L.orc_confidence.argtypes = [vp, ctypes.c_int, vp]
        L.orc_budget.restype = ctypes.c_int
        L.orc_budget.argtypes = [ctypes.c_double, ctypes.c_float, ctypes.c_int, ctypes.c_int]
        L.orc_layer_budget.restype = ctypes.c_int
        L.orc_layer_budget.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, ctypes.c_int]
        L.orc_quantize.restype = None
        L.orc_quantize.argtypes = [vp, ctypes.c_int, vp, vp]
        L.orc_quantize_ch.restype = None
        L.orc_quantize_ch.argtypes = [vp, ctypes.c_int, vp, vp, vp]
        L.orc_channel_exponents.restype = None
        L.orc_channel_exponents.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp]
        L.orc_get_exponents.restype = None
        L.orc_get_exponents.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_ema_update.restype = ctypes.c_float
        L.orc_ema_update.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float]
        L.orc_rank_key.restype = ctypes.c_float
        L.orc_rank_key.argtypes = [ctypes.c_float, ctypes.c_int64]
        L.orc_h2o_update.restype = ctypes.c_float
        L.orc_h2o_update.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_splitmix.restype = ctypes.c_uint64
        L.orc_splitmix.argtypes = [ctypes.c_uint64]
        L.orc_random_key.restype = ctypes.c_float
        L.orc_random_key.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
        L.orc_select.restype = ctypes.c_int
        L.orc_select.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_int, vp]
        L.orc_attention_head.restype = None
        L.orc_attention_head.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_create.restype = vp
        L.orc_create.argtypes = [_P(_Params)]
        L.orc_free.restype = None
        L.orc_free.argtypes = [vp]
        L.orc_set_active.restype = None
        L.orc_set_active.argtypes = [vp, vp]
        L.orc_prefill_lb.restype = ctypes.c_int
        L.orc_prefill_lb.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_int, vp]
        L.orc_set_position.restype = None
        L.orc_set_position.argtypes = [vp, ctypes.c_int64]
        L.orc_step.restype = ctypes.c_int
        L.orc_step.argtypes = [vp] * 8 + [ctypes.c_int, vp, vp, vp]
        L.orc_count.restype = ctypes.c_int
        L.orc_count.argtypes = [vp, ctypes.c_int, ctypes.c_int]
        L.orc_last_keys.restype = ctypes.c_int
        L.orc_last_keys.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                    ctypes.c_int, vp, vp]
        L.orc_get_tokens.restype = ctypes.c_int
        L.orc_get_tokens.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int] + [vp] * 10
        L.orc_half_to_double.restype = ctypes.c_double
        L.orc_half_to_double.argtypes = [ctypes.c_uint16]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _bits16(a):
    """fp16 array -> contiguous uint16 bit view."""
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float16)).view(np.uint16)


# ---------------------------------------------------------------------------
# single operations
# ---------------------------------------------------------------------------

def confidence(z):
    """(c, H_hat, margin, p1, nonfinite) of one logits row."""
    z = _c(z, np.float32)
    comps = np.zeros(4, dtype=np.float64)
    c = lib().orc_confidence(_ptr(z), z.size, _ptr(comps))
    return c, comps[0], comps[1], comps[2], bool(comps[3])


def budget(c, tau, n_low, n_high):
    return lib().orc_budget(float(c), float(tau), int(n_low), int(n_high))


def layer_budget(N, l, L, pyramid_min, P):
    return lib().orc_layer_budget(int(N), int(l), int(L), float(pyramid_min), int(P))


def quantize(x, f=None):
    """INT8 codes and fp32 scale of one fp16 row; f: optional int8 channel
    exponents (the row's channel c is divided by 2^f[c] first)."""
    xb = _bits16(x)
    codes = np.zeros(xb.size, dtype=np.int8)
    scale = np.zeros(1, dtype=np.float32)
    if f is None:
        lib().orc_quantize(_ptr(xb), xb.size, _ptr(codes), _ptr(scale))
    else:
        fb = _c(np.asarray(f).reshape(-1), np.int8)
        assert fb.size == xb.size
        lib().orc_quantize_ch(_ptr(xb), xb.size, _ptr(fb), _ptr(codes), _ptr(scale))
    return codes, np.float32(scale[0])


def channel_exponents(x):
    """int8 channel exponents f[d] of one KV head's prompt rows x [T, d] (fp16)."""
    xb = _bits16(x)
    T, d = (xb.shape if xb.ndim == 2 else (0, xb.shape[-1]))
    f = np.zeros(d, dtype=np.int8)
    lib().orc_channel_exponents(_ptr(xb), T, d, _ptr(f))
    return f


def ema_update(ema, a, beta):
    return np.float32(lib().orc_ema_update(float(ema), float(a), float(beta)))


def rank_key(ema, age):
    return np.float32(lib().orc_rank_key(float(ema), int(age)))


def h2o_update(acc, a):
    return np.float32(lib().orc_h2o_update(float(acc), float(a)))


def splitmix(x):
    """SplitMix64 output function of the word x (the generator's output for
    state x + golden gamma)."""
    return int(lib().orc_splitmix(int(x) & (2**64 - 1)))


def random_key(seed, t, lb, pos):
    return np.float32(lib().orc_random_key(int(seed), int(t), int(lb), int(pos)))


def select(key, pos, prot, N):
    key = _c(key, np.float32)
    pos = _c(pos, np.int32)
    prot = _c(prot, np.uint8)
    keep = np.zeros(key.size, dtype=np.uint8)
    lib().orc_select(key.size, _ptr(key), _ptr(pos), _ptr(prot), int(N), _ptr(keep))
    return keep.astype(bool)


def attention_head(q, k, v):
    """Textbook softmax attention of one head: q [d], k/v [n, d] (float64)."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    n, d = k.shape
    out = np.zeros(d, dtype=np.float64)
    prob = np.zeros(n, dtype=np.float64)
    lib().orc_attention_head(_ptr(q), _ptr(k), _ptr(v), n, d, _ptr(out), _ptr(prob))
    return out, prob


# ---------------------------------------------------------------------------
# whole-cache oracle
# ---------------------------------------------------------------------------

class Oracle:
    """The CONF-KV cache manager of every (layer, sequence), step by step."""

    def __init__(self, L, B, Hq, Hkv, d, V, N_low, N_high, tau, P, W, beta,
                 pyramid_min=1.0, policy=POLICY_CONFKV, seed=0, int8_channel=0):
        self.L, self.B, self.Hq, self.Hkv, self.d, self.V = L, B, Hq, Hkv, d, V
        self.N_low, self.N_high, self.P, self.W = N_low, N_high, P, W
        self.policy = policy
        self.int8_channel = int8_channel
        prm = _Params(L, B, Hq, Hkv, d, V, N_low, N_high, P, W, tau, beta, pyramid_min,
                      policy, int8_channel, seed)
        self._h = lib().orc_create(ctypes.byref(prm))
        if not self._h:
            raise ValueError("oracle: invalid parameters")

    @classmethod
    def for_workload(cls, w, policy=POLICY_CONFKV, seed=0):
        return cls(w.L, w.B, w.Hq, w.Hkv, w.d, w.V, w.N_low, w.N_high, w.tau, w.P,
                   w.W, w.beta, w.pyramid_min, policy, seed, w.int8_channel)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().orc_free(h)
            self._h = None

    def set_active(self, mask):
        m = _c(np.asarray(mask, dtype=np.uint8).reshape(self.L * self.B), np.uint8)
        lib().orc_set_active(self._h, _ptr(m))

    def set_position(self, t):
        lib().orc_set_position(self._h, int(t))

    def prefill_lb(self, l, b, k, v, q_last=None):
        """k, v: [Hkv, T, d] fp16; q_last: [Hq, d] fp16 or None."""
        kb, vb = _bits16(k), _bits16(v)
        T = kb.shape[1] if kb.ndim == 3 else 0
        rc = lib().orc_prefill_lb(self._h, l, b, _ptr(kb), _ptr(vb), T, _ptr(_bits16(q_last)))
        if rc:
            raise ValueError("oracle prefill failed")

    def step(self, logits, q, k_new, v_new, cap=None):
        L, B = self.L, self.B
        cap = cap or max(self.N_low, self.N_high) + 1
        lg = _c(logits, np.float32)
        out = np.zeros((L, B, self.Hq, self.d), dtype=np.float64)
        kept_pos = np.full((L, B, cap), -1, dtype=np.int32)
        kept_count = np.zeros((L, B), dtype=np.int32)
        conf = np.zeros(B, dtype=np.float64)
        bud = np.zeros(B, dtype=np.int32)
        flags = np.zeros(B, dtype=np.int32)
        lib().orc_step(self._h, _ptr(lg), _ptr(_bits16(q)), _ptr(_bits16(k_new)),
                       _ptr(_bits16(v_new)), _ptr(out), _ptr(kept_pos), _ptr(kept_count),
                       cap, _ptr(conf), _ptr(bud), _ptr(flags))
        return dict(out=out, kept_pos=kept_pos, kept_count=kept_count, conf=conf,
                    budget=bud, flags=flags)

    def count(self, l, b):
        return lib().orc_count(self._h, l, b)

    def last_keys(self, l, b):
        cap = self.count(l, b) + 1 + max(self.N_low, self.N_high) + 1 + 100000
        n_max = cap
        key = np.zeros(n_max, dtype=np.float32)
        pos = np.zeros(n_max, dtype=np.int32)
        prot = np.zeros(n_max, dtype=np.uint8)
        bud = ctypes.c_int(0)
        ev = ctypes.c_int(0)
        n = lib().orc_last_keys(self._h, l, b, _ptr(key), _ptr(pos), _ptr(prot), n_max,
                                ctypes.byref(bud), ctypes.byref(ev))
        return dict(key=key[:n], pos=pos[:n], prot=prot[:n].astype(bool),
                    budget=bud.value, evicted=ev.value)

    def exponents(self, l, b):
        """Channel exponents (fk, fv) of (l, b), int8 [Hkv, d] each."""
        fk = np.zeros((self.Hkv, self.d), np.int8)
        fv = np.zeros((self.Hkv, self.d), np.int8)
        lib().orc_get_exponents(self._h, l, b, _ptr(fk), _ptr(fv))
        return fk, fv

    def tokens(self, l, b):
        n = self.count(l, b)
        H, d = self.Hkv, self.d
        r = dict(pos=np.zeros(n, np.int32), is8=np.zeros(n, np.uint8),
                 ema=np.zeros(n, np.float32), a_prev=np.zeros(n, np.float32),
                 k16=np.zeros((n, H, d), np.uint16), v16=np.zeros((n, H, d), np.uint16),
                 k8=np.zeros((n, H, d), np.int8), v8=np.zeros((n, H, d), np.int8),
                 ks=np.zeros((n, H), np.float32), vs=np.zeros((n, H), np.float32))
        lib().orc_get_tokens(self._h, l, b, n, *[_ptr(r[x]) for x in
                             ("pos", "is8", "ema", "a_prev", "k16", "v16", "k8", "v8",
                              "ks", "vs")])
        r["is8"] = r["is8"].astype(bool)
        return r
