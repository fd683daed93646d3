"""ctypes front end of the CPU oracle (liboracle.so).

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline may import this module. The CUDA library never does.
"""
import ctypes
import os
import subprocess

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_DIR, "liboracle.so")
_SRC = [os.path.join(_DIR, "moe_oracle.cpp"), os.path.join(_DIR, "moe_oracle.h")]


def build_cmd():
    return [os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-fPIC",
            "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
            _SRC[0], "-o", _SO]


def build():
    """Compile liboracle.so in-tree if missing or older than its sources."""
    if os.path.exists(_SO) and all(os.path.getmtime(s) <= os.path.getmtime(_SO)
                                   for s in _SRC):
        return
    p = subprocess.run(build_cmd(), capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + p.stdout + p.stderr)


GET_SPAN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                            ctypes.c_int)


class _Layer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("I", ctypes.c_int), ("n_shared", ctypes.c_int),
                ("Is", ctypes.c_int), ("router", ctypes.c_void_p),
                ("shared_gate", ctypes.c_void_p), ("shared_up", ctypes.c_void_p),
                ("shared_down", ctypes.c_void_p), ("get_span", GET_SPAN),
                ("ctx", ctypes.c_void_p), ("layer", ctypes.c_int)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.orc_e2m1_value.argtypes = [ctypes.c_uint8]; L.orc_e2m1_value.restype = dbl
        L.orc_e8m0_value.argtypes = [ctypes.c_uint8]; L.orc_e8m0_value.restype = dbl
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]; L.orc_bf16_to_f64.restype = dbl
        L.orc_f64_to_bf16.argtypes = [dbl]; L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_span_bytes.argtypes = [i32, i32]; L.orc_span_bytes.restype = ctypes.c_size_t
        L.orc_span_offsets.argtypes = [i32, i32, vp]
        L.orc_mx_dequant.argtypes = [vp, vp, i32, i32, vp]
        L.orc_mx_gemv.argtypes = [vp, vp, i32, i32, vp, vp]
        L.orc_router_logits.argtypes = [vp, i32, i32, vp, i32, vp]
        L.orc_topk_softmax.argtypes = [vp, i32, i32, i32, vp, vp]
        L.orc_silu.argtypes = [dbl]; L.orc_silu.restype = dbl
        L.orc_expert_gateup.argtypes = [vp, i32, i32, vp, vp]
        L.orc_expert_down.argtypes = [vp, i32, i32, vp, vp]
        L.orc_expert_ffn.argtypes = [vp, i32, i32, vp, vp]
        L.orc_shared_ffn.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.orc_group.argtypes = [vp, i32, i32, i32, vp, vp, vp]; L.orc_group.restype = i32
        L.orc_rmsnorm_bf16.argtypes = [vp, i32, i32, dbl, vp]
        L.orc_moe_layer.argtypes = [ctypes.POINTER(_Layer), vp, i32, vp, vp, vp,
                                    vp, vp, vp, vp]
        L.orc_moe_layer.restype = i32
        L.orc_moe_stack.argtypes = [ctypes.POINTER(_Layer), i32, vp, i32, dbl, vp,
                                    vp, vp, vp, vp]
        L.orc_moe_stack.restype = i32
        L.orc_e4m3_value.argtypes = [ctypes.c_uint8]; L.orc_e4m3_value.restype = dbl
        L.orc_e4m3_from_f64.argtypes = [dbl]; L.orc_e4m3_from_f64.restype = ctypes.c_uint8
        L.orc_mxfp8_quantize.argtypes = [vp, i32, i32, vp, vp]
        L.orc_mxfp8_dequant.argtypes = [vp, vp, i32, i32, vp]
        L.orc_num_threads.restype = i32
        L.orc_set_num_threads.argtypes = [i32]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- formats ----------------------------------------------------------------

def e2m1_value(code):
    return lib().orc_e2m1_value(code)


def e8m0_value(e):
    return lib().orc_e8m0_value(e)


def bf16_to_f64(b):
    return lib().orc_bf16_to_f64(int(b))


def f64_to_bf16(v):
    return lib().orc_f64_to_bf16(float(v))


def span_bytes(H, I):
    return lib().orc_span_bytes(H, I)


def span_offsets(H, I):
    off = np.zeros(6, dtype=np.uint64)
    lib().orc_span_offsets(H, I, _p(off))
    return [int(v) for v in off]


def span_tensors(span, H, I):
    """Views (gate_q, gate_s, up_q, up_s, down_q, down_s) of a canonical span."""
    o = span_offsets(H, I) + [span_bytes(H, I)]
    shapes = [(I, H // 2), (I, H // 32), (I, H // 2), (I, H // 32),
              (H, I // 2), (H, I // 32)]
    return [span[o[i]:o[i + 1]].reshape(shapes[i]) for i in range(6)]


# ---- steps ------------------------------------------------------------------

def mx_dequant(q, s):
    q = _c(q, np.uint8); s = _c(s, np.uint8)
    rows, cols = q.shape[0], q.shape[1] * 2
    W = np.empty((rows, cols), dtype=np.float64)
    lib().orc_mx_dequant(_p(q), _p(s), rows, cols, _p(W))
    return W


def mx_gemv(q, s, x):
    q = _c(q, np.uint8); s = _c(s, np.uint8); x = _c(x, np.float64)
    rows, cols = q.shape[0], q.shape[1] * 2
    y = np.empty(rows, dtype=np.float64)
    lib().orc_mx_gemv(_p(q), _p(s), rows, cols, _p(x), _p(y))
    return y


def router_logits(Wr, x_bf16):
    Wr = _c(Wr, np.float32); x = _c(x_bf16, np.uint16)
    E, H = Wr.shape
    T = x.size // H
    out = np.empty((T, E), dtype=np.float64)
    lib().orc_router_logits(_p(Wr), E, H, _p(x), T, _p(out))
    return out


def topk_softmax(logits, k):
    logits = _c(logits, np.float64)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().orc_topk_softmax(_p(logits), T, E, k, _p(ids), _p(w))
    return ids, w


def silu(g):
    return lib().orc_silu(float(g))


def expert_gateup(span, H, I, x):
    span = _c(span, np.uint8); x = _c(x, np.float64)
    h = np.empty(I, dtype=np.float64)
    lib().orc_expert_gateup(_p(span), H, I, _p(x), _p(h))
    return h


def expert_down(span, H, I, h):
    span = _c(span, np.uint8); h = _c(h, np.float64)
    y = np.empty(H, dtype=np.float64)
    lib().orc_expert_down(_p(span), H, I, _p(h), _p(y))
    return y


def expert_ffn(span, H, I, x):
    span = _c(span, np.uint8); x = _c(x, np.float64)
    y = np.empty(H, dtype=np.float64)
    lib().orc_expert_ffn(_p(span), H, I, _p(x), _p(y))
    return y


def shared_ffn(gate, up, down, x):
    gate = _c(gate, np.uint16); up = _c(up, np.uint16); down = _c(down, np.uint16)
    x = _c(x, np.float64)
    Is, H = gate.shape
    y = np.empty(H, dtype=np.float64)
    lib().orc_shared_ffn(_p(gate), _p(up), _p(down), H, Is, _p(x), _p(y))
    return y


def group(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offs = np.empty(E + 1, dtype=np.int32)
    tok = np.empty(T * k, dtype=np.int32)
    slot = np.empty(T * k, dtype=np.int32)
    n = lib().orc_group(_p(ids), T, k, E, _p(offs), _p(tok), _p(slot))
    return offs, tok, slot, n


def rmsnorm_bf16(x, eps):
    x = _c(x, np.uint16)
    T, H = x.shape
    out = np.empty_like(x)
    lib().orc_rmsnorm_bf16(_p(x), T, H, eps, _p(out))
    return out


# ---- MXFP8 activations (the lossy variant) ----------------------------------

def e4m3_value(code):
    return lib().orc_e4m3_value(code)


def e4m3_from_f64(v):
    return lib().orc_e4m3_from_f64(float(v))


def mxfp8_quantize(v):
    """Rows of v (last dimension a multiple of 32) -> (codes u8, scales u8)."""
    v = _c(v, np.float64)
    shp = v.shape
    n = shp[-1]
    rows = v.size // n
    codes = np.empty(shp, dtype=np.uint8)
    scales = np.empty(shp[:-1] + (n // 32,), dtype=np.uint8)
    lib().orc_mxfp8_quantize(_p(v), rows, n, _p(codes), _p(scales))
    return codes, scales


def mxfp8_dequant(codes, scales):
    codes = _c(codes, np.uint8); scales = _c(scales, np.uint8)
    n = codes.shape[-1]
    rows = codes.size // n
    v = np.empty(codes.shape, dtype=np.float64)
    lib().orc_mxfp8_dequant(_p(codes), _p(scales), rows, n, _p(v))
    return v


def mxfp8_round(v):
    """The values the MXFP8 format holds for v (quantise, then dequantise)."""
    return mxfp8_dequant(*mxfp8_quantize(v))


def moe_layer_mxfp8(layer, x_bf16, residual=None, h_in=None):
    """The layer with MXFP8 activations into the routed experts: every routed
    expert takes x rounded to MXFP8, and its down projection takes h rounded
    to MXFP8; router and shared experts are exact. h_in (optional, [T*k][I]
    in the order t*k + j) replaces the oracle's own h before its rounding, so
    that a caller can feed the h of the device (the rounding then decides on
    the same values). Returns dict(out, ids, w, routed, shared, h)."""
    L = layer.s
    H, I, k = L.H, L.I, L.k
    x = _c(x_bf16, np.uint16).reshape(-1, H)
    T = x.shape[0]
    ref = moe_layer(layer, x, residual)
    ids, w = ref["ids"], ref["w"]
    xd = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xq = mxfp8_round(xd)
    routed = np.zeros((T, H))
    hs = np.empty((T * k, I))
    for t in range(T):
        for j in range(k):
            span = layer._spans(L.layer, int(ids[t, j]))
            h = expert_gateup(span, H, I, xq[t])
            hs[t * k + j] = h
            hh = h if h_in is None else np.asarray(h_in[t * k + j], dtype=np.float64)
            routed[t] += w[t, j] * expert_down(span, H, I, mxfp8_round(hh[None, :])[0])
    res = 0.0 if residual is None else (
        (_c(residual, np.uint16).reshape(T, H).astype(np.uint32) << 16)
        .view(np.float32).astype(np.float64))
    out = res + (routed + ref["shared"])
    return dict(out=out, ids=ids, w=w, routed=routed, shared=ref["shared"], h=hs)


# ---- layer / stack ----------------------------------------------------------

class Layer:
    """One MoE layer's weights for the oracle. `spans` is a callable
    (layer, expert) -> canonical span (np.uint8), called once per needed
    expert."""

    def __init__(self, H, E, k, I, Is, router, shared, spans, layer=0):
        self.keep = []
        self.router = _c(router, np.float32)
        sg = [_c(s[0], np.uint16) for s in shared]
        su = [_c(s[1], np.uint16) for s in shared]
        sd = [_c(s[2], np.uint16) for s in shared]
        self.keep += [self.router] + sg + su + sd
        arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(
            *[x.ctypes.data for x in xs])
        self._sg, self._su, self._sd = arr(sg), arr(su), arr(sd)
        self._spans = spans
        self._cache = {}

        def get_span(ctx, lyr, e):
            try:
                a = self._cache.get((lyr, e))
                if a is None:
                    a = _c(self._spans(lyr, e), np.uint8)
                    self._cache[(lyr, e)] = a
                return a.ctypes.data
            except Exception:  # a NULL tells the oracle the span is missing
                return None

        self._cb = GET_SPAN(get_span)
        self.s = _Layer(H, E, k, I, len(shared), Is, self.router.ctypes.data,
                        ctypes.cast(self._sg, ctypes.c_void_p),
                        ctypes.cast(self._su, ctypes.c_void_p),
                        ctypes.cast(self._sd, ctypes.c_void_p), self._cb, None,
                        layer)

    def clear_cache(self):
        self._cache.clear()


def moe_layer(layer, x_bf16, residual=None):
    """Returns dict(out, ids, w, logits, routed, shared) for tokens x [T, H]."""
    L = layer.s
    x = _c(x_bf16, np.uint16).reshape(-1, L.H)
    T = x.shape[0]
    res = None if residual is None else _c(residual, np.uint16).reshape(T, L.H)
    out = np.empty((T, L.H)); routed = np.empty((T, L.H)); shared = np.empty((T, L.H))
    ids = np.empty((T, L.k), dtype=np.int32); w = np.empty((T, L.k))
    logits = np.empty((T, L.E))
    rc = lib().orc_moe_layer(ctypes.byref(L), _p(x), T, _p(res), _p(out), _p(ids),
                             _p(w), _p(logits), _p(routed), _p(shared))
    if rc:
        raise RuntimeError("oracle: an expert span was unavailable")
    return dict(out=out, ids=ids, w=w, logits=logits, routed=routed,
                shared=shared)


def moe_stack(layers, x_bf16, eps):
    H, k = layers[0].s.H, layers[0].s.k
    x = _c(x_bf16, np.uint16).reshape(-1, H)
    T, nl = x.shape[0], len(layers)
    arr = (_Layer * nl)(*[l.s for l in layers])
    x_out = np.empty_like(x); last = np.empty((T, H))
    E = layers[0].s.E
    ids = np.empty((nl, T, k), dtype=np.int32); w = np.empty((nl, T, k))
    logits = np.empty((nl, T, E))
    rc = lib().orc_moe_stack(arr, nl, _p(x), T, eps, _p(x_out), _p(last), _p(ids),
                             _p(w), _p(logits))
    if rc:
        raise RuntimeError("oracle: an expert span was unavailable")
    return dict(x=x_out, last=last, ids=ids, w=w, logits=logits)


def num_threads():
    return lib().orc_num_threads()


def set_num_threads(n):
    lib().orc_set_num_threads(n)
