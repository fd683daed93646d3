"""ctypes front end of the seeded generator (host: libsynth.so, device:
libsynth_dev.so). See synth.h for the definition of every stream."""
import ctypes
import math
import os
import subprocess

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_DIR, "libsynth.so")
_DEV_SO = os.path.join(_DIR, "libsynth_dev.so")

KIND_ROUTER = 1
KIND_SHARED_GATE = 2
KIND_SHARED_UP = 3
KIND_SHARED_DOWN = 4
KIND_X = 5
KIND_RESIDUAL = 6
KIND_X_STREAM = 7
KIND_EXPERT_BASE = 16

# redraw sub-seeds per token (tokens whose routing gap is too small are redrawn)
REDRAWS_PER_TOKEN = 64


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def host_build_cmd():
    src = os.path.join(_DIR, "synth.c")
    return ([os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-fPIC", "-shared",
             "-fopenmp", "-ffp-contract=off", "-fno-fast-math", src, "-o",
             _HOST_SO, "-lm"], [src, os.path.join(_DIR, "synth.h")], _HOST_SO)


def dev_build_cmd():
    src = os.path.join(_DIR, "synth_dev.cu")
    return (["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC",
             "-gencode", "arch=compute_103a,code=sm_103a", src, "-o", _DEV_SO],
            [src], _DEV_SO)


def build(device=True):
    """Compile the generator libraries in-tree (skips up-to-date ones)."""
    cmds = [host_build_cmd()] + ([dev_build_cmd()] if device else [])
    procs = []
    for cmd, srcs, out in cmds:
        if _stale(out, srcs):
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("build failed: %s\n%s" % (" ".join(cmd),
                                                         out.decode()))


_host = None
_dev = None


def _lib():
    global _host
    if _host is None:
        if not os.path.exists(_HOST_SO):
            build(device=False)
        L = ctypes.CDLL(_HOST_SO)
        u64, u32, i32 = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        vp, dbl = ctypes.c_void_p, ctypes.c_double
        L.synth_mix64.argtypes = [u64]; L.synth_mix64.restype = u64
        L.synth_at.argtypes = [u64, u64]; L.synth_at.restype = u64
        L.synth_key.argtypes = [u64, u32, u32, u32, u64]; L.synth_key.restype = u64
        L.synth_span_bytes.argtypes = [i32, i32]; L.synth_span_bytes.restype = ctypes.c_size_t
        L.synth_expert_spans.argtypes = [u64, u32, u32, u32, u32, i32, i32, vp]
        for f in (L.synth_normal_f64, L.synth_normal_f32, L.synth_normal_bf16):
            f.argtypes = [u64, u64, u64, dbl, vp]
        L.synth_words.argtypes = [u64, u64, u64, vp]
        L.synth_num_threads.restype = i32
        _host = L
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_DEV_SO):
            raise RuntimeError("libsynth_dev.so is not built (run build())")
        L = ctypes.CDLL(_DEV_SO)
        L.synth_dev_expert_spans.argtypes = [
            ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
            ctypes.c_uint32, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p]
        L.synth_dev_expert_spans.restype = ctypes.c_int
        _dev = L
    return _dev


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def mix64(z):
    return _lib().synth_mix64(z)


def at(key, i):
    return _lib().synth_at(key, i)


def key(seed, cfg, layer, kind, index):
    return _lib().synth_key(seed, cfg, layer, kind, index)


def span_bytes(H, I):
    return _lib().synth_span_bytes(H, I)


def words(k, first, n):
    out = np.empty(n, dtype=np.uint64)
    _lib().synth_words(k, first, n, _ptr(out))
    return out


def expert_spans(seed, cfg, layer, e0, n, H, I):
    """n canonical expert spans as a uint8 array [n, span_bytes]."""
    out = np.empty((n, span_bytes(H, I)), dtype=np.uint8)
    _lib().synth_expert_spans(seed, cfg, layer, e0, n, H, I, _ptr(out))
    return out


def normal_f64(k, n, sigma, first=0):
    out = np.empty(n, dtype=np.float64)
    _lib().synth_normal_f64(k, first, n, sigma, _ptr(out))
    return out


def normal_f32(k, n, sigma, first=0):
    out = np.empty(n, dtype=np.float32)
    _lib().synth_normal_f32(k, first, n, sigma, _ptr(out))
    return out


def normal_bf16(k, n, sigma, first=0):
    """bf16 bit patterns (uint16)."""
    out = np.empty(n, dtype=np.uint16)
    _lib().synth_normal_bf16(k, first, n, sigma, _ptr(out))
    return out


# ---- the workload tensors -------------------------------------------------

def router(seed, cfg, layer, E, H):
    """fp32 [E, H] ~ N(0, 1/H): logits of a N(0,1) token are ~N(0,1), so the
    expected expert load is uniform."""
    k = key(seed, cfg, layer, KIND_ROUTER, 0)
    return normal_f32(k, E * H, 1.0 / math.sqrt(H)).reshape(E, H)


def shared(seed, cfg, layer, s, H, Is, sigma=0.02):
    """bf16 bits: gate [Is, H], up [Is, H], down [H, Is] of shared expert s."""
    g = normal_bf16(key(seed, cfg, layer, KIND_SHARED_GATE, s), Is * H, sigma)
    u = normal_bf16(key(seed, cfg, layer, KIND_SHARED_UP, s), Is * H, sigma)
    d = normal_bf16(key(seed, cfg, layer, KIND_SHARED_DOWN, s), H * Is, sigma)
    return g.reshape(Is, H), u.reshape(Is, H), d.reshape(H, Is)


def token(seed, cfg, token_id, H, redraw=0, kind=KIND_X):
    """bf16 bits [H] ~ N(0, 1) of one token (redraw r gives an independent
    replacement draw for the same token slot)."""
    if not 0 <= redraw < REDRAWS_PER_TOKEN:
        raise ValueError("redraw out of range")
    k = key(seed, cfg, 0, kind, token_id * REDRAWS_PER_TOKEN + redraw)
    return normal_bf16(k, H, 1.0)


def f64_to_bf16_bits(a):
    """Round fp64 values to bf16 (through fp32, nearest-even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def token_stream(seed, cfg, first, n, H, rho, stream=0):
    """bf16 bits [n, H]: consecutive tokens of a stream with temporal
    correlation, x_0 = z_0 and x_i = rho x_(i-1) + sqrt(1 - rho^2) z_i with
    z_i ~ N(0, 1) i.i.d. (a stationary AR(1) process per coordinate, so each
    token is N(0, 1) and neighbours have correlation rho). Token i of the
    stream starting at `first` is the same whatever n is. rho = 0 gives
    independent tokens. `stream` selects one of independent streams (it takes
    the layer field of the key)."""
    if not 0.0 <= rho < 1.0:
        raise ValueError("rho must be in [0, 1)")
    c = math.sqrt(1.0 - rho * rho)
    x = normal_f64(key(seed, cfg, stream, KIND_X_STREAM, 0), H, 1.0)
    out = np.empty((n, H), dtype=np.uint16)
    for i in range(first + n):
        if i:
            x = rho * x + c * normal_f64(key(seed, cfg, stream, KIND_X_STREAM, i), H, 1.0)
        if i >= first:
            out[i - first] = f64_to_bf16_bits(x)
    return out


def dev_expert_spans(seed, cfg, layer, e0, n, H, I, dst_ptr, stream_ptr=0):
    """Write n canonical spans to device memory at dst_ptr (device pointer)."""
    rc = _dev_lib().synth_dev_expert_spans(seed, cfg, layer, e0, n, H, I,
                                           ctypes.c_void_p(dst_ptr),
                                           ctypes.c_void_p(stream_ptr))
    if rc != 0:
        raise RuntimeError("synth_dev_expert_spans failed: cudaError %d" % rc)


def num_threads():
    return _lib().synth_num_threads()
