"""GPU twin of the seeded input generator (fills torch CUDA tensors in place).

Bit-identical to ``synth.gen`` (checked by a GPU test); used to create inputs
too large to build on the host, e.g. multi-GB prefills.
"""
import ctypes
import os
import shutil
import subprocess

from . import gen

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth.cu")
_LIB = os.path.join(_HERE, "_build", "libconfkv_synth.so")
_lib = None


def build(force=False):
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _SRC], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.synth_fill_f16.restype = ctypes.c_int
        L.synth_fill_f16.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_ulonglong,
                                     ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
                                     ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_logits.restype = ctypes.c_int
        L.synth_fill_logits.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_ulonglong,
                                        ctypes.c_double, ctypes.c_void_p]
        L.synth_read_probe.restype = ctypes.c_int
        L.synth_read_probe.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p,
                                       ctypes.c_int, ctypes.c_void_p]
        _lib = L
    return _lib


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_f16(t, seed, kind, step, heavy=False, inner=1, tlen=1, pos0=0):
    """t: contiguous float16 CUDA tensor = the full tensor of stream (seed, kind, step)."""
    import torch
    assert t.is_cuda and t.dtype == torch.float16 and t.is_contiguous()
    rc = lib().synth_fill_f16(ctypes.c_void_p(t.data_ptr()), t.numel(),
                              gen.stream_key(seed, kind, step), inner, tlen, pos0,
                              1 if heavy else 0, _stream())
    if rc:
        raise RuntimeError(f"synth_fill_f16 failed ({rc})")
    return t


def fill_logits(t, seed, step, temperature):
    import torch
    assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
    rc = lib().synth_fill_logits(ctypes.c_void_p(t.data_ptr()), t.numel(),
                                 gen.stream_key(seed, gen.KIND_LOGITS, step),
                                 float(temperature), _stream())
    if rc:
        raise RuntimeError(f"synth_fill_logits failed ({rc})")
    return t


# ---- workload tensors on the device ----

def step_inputs(w, s, out=None):
    """(logits, q, k_new, v_new) of decode step s, filled on the current device."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = (torch.empty(w.B, w.V, dtype=torch.float32, device=dev),
               torch.empty(w.L, w.B, w.Hq, w.d, dtype=torch.float16, device=dev),
               torch.empty(w.L, w.B, w.Hkv, w.d, dtype=torch.float16, device=dev),
               torch.empty(w.L, w.B, w.Hkv, w.d, dtype=torch.float16, device=dev))
    lg, q, k, v = out
    fill_logits(lg, w.seed, s, w.temperature(s))
    fill_f16(q, w.seed, gen.KIND_Q, s)
    fill_f16(k, w.seed, gen.KIND_KNEW, s, heavy=True, inner=w.d, tlen=1, pos0=w.position(s))
    fill_f16(v, w.seed, gen.KIND_VNEW, s)
    return out


def prefill_kv(w):
    """k, v [L, B, Hkv, T, d] on the device, needles included."""
    import numpy as np
    import torch
    from . import workloads as wl
    dev = torch.device("cuda", torch.cuda.current_device())
    shape = (w.L, w.B, w.Hkv, w.prefill, w.d)
    k = torch.empty(shape, dtype=torch.float16, device=dev)
    v = torch.empty(shape, dtype=torch.float16, device=dev)
    fill_f16(k, w.seed, gen.KIND_KPRE, 0, heavy=True, inner=w.d, tlen=w.prefill, pos0=0)
    fill_f16(v, w.seed, gen.KIND_VPRE, 0)
    if w.needles:
        for l in range(w.L):
            for b in range(w.B):
                pos = gen.needle_positions(w.seed, b, w.prefill, w.W, w.needles)
                rows = np.zeros((w.Hkv, w.prefill, w.d), np.float16)
                n = w.Hkv * w.prefill * w.d
                lo = (l * w.B + b) * n
                # only the needle rows are needed: regenerate them on the host
                for h in range(w.Hkv):
                    for p in pos:
                        a = lo + (h * w.prefill + int(p)) * w.d
                        rows[h, p] = gen.gen_f16(w.seed, gen.KIND_KPRE, 0, shape, a, a + w.d,
                                                 inner=w.d, tlen=w.prefill, heavy=True)
                pos_, vals = wl.needle_keys_lb(w, l, b, rows)
                t = torch.from_numpy(vals).to(dev)                    # [n, Hkv, d]
                k[l, b][:, torch.from_numpy(pos_).to(dev), :] = t.permute(1, 0, 2)
    return k, v


def read_bandwidth_gbs(gib=4, reps=5):
    """Best-of-`reps` HBM read rate (GB/s) of one pass over a `gib` GiB buffer
    (CUDA events around each pass; the buffer is 30x the L2)."""
    import torch
    n = int(gib * (1 << 30))
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    sink = torch.zeros(64, dtype=torch.int32, device="cuda")
    sms = torch.cuda.get_device_properties(buf.device).multi_processor_count
    best = 0.0
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        rc = lib().synth_read_probe(ctypes.c_void_p(buf.data_ptr()), n,
                                    ctypes.c_void_p(sink.data_ptr()), sms * 8, _stream())
        e1.record()
        torch.cuda.synchronize()
        if rc:
            raise RuntimeError(f"synth_read_probe failed ({rc})")
        best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del buf
    return best
