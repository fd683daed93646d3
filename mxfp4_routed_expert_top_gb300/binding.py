"""Thin ctypes binding of libdfmoe.so (include/df_moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. torch tensors are accepted wherever the C call takes a pointer (their
data_ptr() is passed); streams are torch.cuda.Stream objects or raw handles.
There is no fallback: if the library is missing this module raises.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdfmoe.so")

OK, EINVAL, ENOMEM, ECUDA, ESTATE, ERANGE, ETIMEOUT, EDEVICE = 0, -1, -2, -3, -4, -5, -6, -7
STACK_RMSNORM_RESIDUAL = 1
PREFILL_MMA_SYNC = 4
MXFP8_ACT = 8
PLANES = 16
KERNEL_KINDS = 18

# every symbol the header declares (checked by the CPU tests)
SYMBOLS = [
    "df_moe_create", "df_moe_destroy", "df_moe_last_error",
    "df_moe_expert_span_bytes", "df_moe_span_bytes_for", "df_moe_load_experts",
    "df_moe_forward", "df_moe_forward_trace", "df_moe_forward_host", "df_moe_sync",
    "df_moe_step_router", "df_moe_step_topk", "df_moe_step_group",
    "df_moe_step_expert_gateup", "df_moe_step_expert_down",
    "df_moe_step_shared", "df_moe_step_rmsnorm", "df_moe_read_expert_span",
    "df_moe_timing_enable", "df_moe_timing_reset", "df_moe_timing_get",
    "df_moe_last_launch_count", "df_moe_route_noalloc",
    "df_moe_graph_create", "df_moe_graph_launch", "df_moe_graph_launch_count",
    "df_moe_graph_destroy", "df_moe_stream_read", "df_moe_create_cached",
    "df_moe_cache_stats", "df_moe_test_drop_arrival", "df_moe_step_mxfp8",
]


class DfMoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("df_moe error %d: %s" % (code, msg))
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("router", ctypes.c_void_p), ("experts", ctypes.c_void_p),
                ("expert_begin", ctypes.c_int32), ("expert_count", ctypes.c_int32),
                ("shared_gate", ctypes.c_void_p), ("shared_up", ctypes.c_void_p),
                ("shared_down", ctypes.c_void_p), ("src_is_device", ctypes.c_int32)]


_lib = None


def lib():
    """Loads libdfmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libdfmoe.so is not built; run __graft_entry__.build() "
                              "or python -m mxfp4_routed_expert_top_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.df_moe_create.argtypes = [ctypes.POINTER(Config), ctypes.c_int,
                                    ctypes.POINTER(vp)]
        L.df_moe_destroy.argtypes = [vp]; L.df_moe_destroy.restype = None
        L.df_moe_last_error.argtypes = [vp]; L.df_moe_last_error.restype = ctypes.c_char_p
        L.df_moe_expert_span_bytes.argtypes = [vp]
        L.df_moe_expert_span_bytes.restype = ctypes.c_size_t
        L.df_moe_span_bytes_for.argtypes = [i32, i32]
        L.df_moe_span_bytes_for.restype = ctypes.c_size_t
        L.df_moe_load_experts.argtypes = [vp, i32, ctypes.POINTER(LayerWeights), vp]
        L.df_moe_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.df_moe_forward_trace.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
        L.df_moe_forward_host.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.df_moe_sync.argtypes = [vp, vp]
        L.df_moe_step_router.argtypes = [vp, i32, vp, i32, vp, vp]
        L.df_moe_step_topk.argtypes = [vp, vp, i32, vp, vp, vp]
        L.df_moe_step_group.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
        L.df_moe_step_expert_gateup.argtypes = [vp, i32, vp, i32, vp, vp, vp]
        L.df_moe_step_expert_down.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp]
        L.df_moe_step_shared.argtypes = [vp, i32, vp, i32, vp, vp]
        L.df_moe_step_rmsnorm.argtypes = [vp, vp, i32, vp, vp]
        L.df_moe_step_mxfp8.argtypes = [vp, vp, i32, i32, vp, vp, vp]
        L.df_moe_read_expert_span.argtypes = [vp, i32, i32, vp]
        L.df_moe_timing_enable.argtypes = [vp, ctypes.c_int]
        L.df_moe_timing_reset.argtypes = [vp]
        L.df_moe_timing_get.argtypes = [vp, ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                        ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
        L.df_moe_last_launch_count.argtypes = [vp]
        L.df_moe_route_noalloc.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, vp]
        L.df_moe_graph_create.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp,
                                          ctypes.POINTER(ctypes.c_void_p)]
        L.df_moe_graph_launch.argtypes = [vp, vp]
        L.df_moe_graph_launch_count.argtypes = [vp]
        L.df_moe_graph_destroy.argtypes = [vp]; L.df_moe_graph_destroy.restype = None
        L.df_moe_stream_read.argtypes = [vp, ctypes.c_size_t, vp, vp]
        L.df_moe_create_cached.argtypes = [ctypes.POINTER(Config), ctypes.c_int, i32,
                                           ctypes.POINTER(ctypes.c_void_p)]
        L.df_moe_cache_stats.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                         ctypes.POINTER(i64)]
        for name in SYMBOLS:
            f = getattr(L, name)
            if f.restype is ctypes.c_int:  # default
                f.restype = ctypes.c_int
        _lib = L
    return _lib


def span_bytes_for(H, I):
    return lib().df_moe_span_bytes_for(H, I)


def route_noalloc(router, E, H, x, T, k, ids, weights, stream=None):
    """Router + top-k with no device allocation (df_moe_route_noalloc): for
    callers that must not allocate, e.g. an engine whose memory pools already
    own all of HBM. Same kernels and results as step_router + step_topk."""
    rc = lib().df_moe_route_noalloc(_ptr(router), E, H, _ptr(x), T, k, _ptr(ids),
                                    _ptr(weights), _stream(stream))
    if rc != OK:
        raise DfMoeError(rc, lib().df_moe_last_error(None).decode())


def _ptr(a):
    """Pointer of a torch tensor / numpy array / int / None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        return a.ctypes.data
    raise TypeError("cannot take the address of %r" % type(a))


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


class MoE:
    """Owns one df_moe handle. Methods mirror the C calls (df_moe_ prefix
    dropped) and raise DfMoeError on failure."""

    def __init__(self, hidden, n_experts, top_k, inter, n_shared, shared_inter,
                 n_layers=1, max_tokens=1, rms_eps=1e-6, flags=0, device=0, cache_slots=0):
        """cache_slots > 0: experts in pinned host memory, that many a layer
        in HBM (df_moe_create_cached)."""
        self.cfg = Config(hidden, n_experts, top_k, inter, n_shared, shared_inter,
                          n_layers, max_tokens, rms_eps, flags)
        h = ctypes.c_void_p()
        if cache_slots:
            rc = lib().df_moe_create_cached(ctypes.byref(self.cfg), device, cache_slots,
                                            ctypes.byref(h))
        else:
            rc = lib().df_moe_create(ctypes.byref(self.cfg), device, ctypes.byref(h))
        if rc != OK:
            raise DfMoeError(rc, lib().df_moe_last_error(None).decode())
        self.h = h
        self.device = device

    def close(self):
        if getattr(self, "h", None):
            lib().df_moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def _check(self, rc):
        if rc != OK:
            raise DfMoeError(rc, lib().df_moe_last_error(self.h).decode())

    @property
    def span_bytes(self):
        return lib().df_moe_expert_span_bytes(self.h)

    def load_experts(self, layer, router=None, experts=None, expert_begin=0,
                     expert_count=0, shared=None, src_is_device=False, stream=None):
        """shared: list of (gate, up, down) per shared expert (or None)."""
        keep = []
        sg = su = sd = None
        if shared:
            n = len(shared)
            arr = lambda i: (ctypes.c_void_p * n)(*[_ptr(s[i]) for s in shared])
            sg, su, sd = arr(0), arr(1), arr(2)
            keep += [sg, su, sd]
        w = LayerWeights(_ptr(router), _ptr(experts), expert_begin, expert_count,
                         ctypes.cast(sg, ctypes.c_void_p) if sg else None,
                         ctypes.cast(su, ctypes.c_void_p) if su else None,
                         ctypes.cast(sd, ctypes.c_void_p) if sd else None,
                         1 if src_is_device else 0)
        self._check(lib().df_moe_load_experts(self.h, layer, ctypes.byref(w),
                                              _stream(stream)))

    def forward(self, x, T, out, ids, weights, residual=None, out_f32=None,
                stream=None):
        self._check(lib().df_moe_forward(self.h, _ptr(x), T, _ptr(residual), _ptr(out),
                                         _ptr(out_f32), _ptr(ids), _ptr(weights),
                                         _stream(stream)))

    def forward_trace(self, x, T, out, ids, weights, trace_x=None, trace_xn=None,
                      out_f32=None, stream=None):
        """Stack mode: forward that also records each layer's input x and its
        normalised form xn ([L][T][H] bf16 device buffers)."""
        self._check(lib().df_moe_forward_trace(self.h, _ptr(x), T, _ptr(out), _ptr(out_f32),
                                               _ptr(ids), _ptr(weights), _ptr(trace_x),
                                               _ptr(trace_xn), _stream(stream)))

    def forward_host(self, x, T, out, ids=None, weights=None, residual=None,
                     out_f32=None, stream=None):
        self._check(lib().df_moe_forward_host(self.h, _ptr(x), T, _ptr(residual),
                                              _ptr(out), _ptr(out_f32), _ptr(ids),
                                              _ptr(weights), _stream(stream)))

    def sync(self, stream=None):
        self._check(lib().df_moe_sync(self.h, _stream(stream)))

    def test_drop_arrival(self):
        """Test hook: the next forward's gate/up phase leaves one pipeline
        stage unfilled, so a bounded device wait runs out (ETIMEOUT)."""
        self._check(lib().df_moe_test_drop_arrival(self.h))

    def step_router(self, layer, x, T, logits, stream=None):
        self._check(lib().df_moe_step_router(self.h, layer, _ptr(x), T, _ptr(logits),
                                             _stream(stream)))

    def step_topk(self, logits, T, ids, weights, stream=None):
        self._check(lib().df_moe_step_topk(self.h, _ptr(logits), T, _ptr(ids),
                                           _ptr(weights), _stream(stream)))

    def step_group(self, ids, T, offs, tok, slot, n_union, stream=None):
        self._check(lib().df_moe_step_group(self.h, _ptr(ids), T, _ptr(offs), _ptr(tok),
                                            _ptr(slot), _ptr(n_union), _stream(stream)))

    def step_expert_gateup(self, layer, x, T, ids, hbuf, stream=None):
        self._check(lib().df_moe_step_expert_gateup(self.h, layer, _ptr(x), T, _ptr(ids),
                                                    _ptr(hbuf), _stream(stream)))

    def step_expert_down(self, layer, hbuf, T, ids, weights, y, stream=None):
        self._check(lib().df_moe_step_expert_down(self.h, layer, _ptr(hbuf), T, _ptr(ids),
                                                  _ptr(weights), _ptr(y), _stream(stream)))

    def step_shared(self, layer, x, T, y, stream=None):
        self._check(lib().df_moe_step_shared(self.h, layer, _ptr(x), T, _ptr(y),
                                             _stream(stream)))

    def step_rmsnorm(self, x, T, xn, stream=None):
        self._check(lib().df_moe_step_rmsnorm(self.h, _ptr(x), T, _ptr(xn),
                                              _stream(stream)))

    def step_mxfp8(self, v, rows, n, codes, scales, stream=None):
        """The library's MXFP8 rounding of fp32 rows v [rows][n]: E4M3 codes
        [rows][n] and E8M0 scales [rows][n/32]."""
        self._check(lib().df_moe_step_mxfp8(self.h, _ptr(v), rows, n, _ptr(codes), _ptr(scales),
                                            _stream(stream)))

    def read_expert_span(self, layer, expert, dst):
        self._check(lib().df_moe_read_expert_span(self.h, layer, expert, _ptr(dst)))

    def timing_enable(self, on=True):
        self._check(lib().df_moe_timing_enable(self.h, 1 if on else 0))

    def timing_reset(self):
        self._check(lib().df_moe_timing_reset(self.h))

    def timing(self):
        """{kernel kind name: (launches, total_ms)} since the last reset."""
        out = {}
        for kind in range(KERNEL_KINDS):
            name = ctypes.c_char_p()
            n = ctypes.c_int64()
            ms = ctypes.c_double()
            self._check(lib().df_moe_timing_get(self.h, kind, ctypes.byref(name),
                                                ctypes.byref(n), ctypes.byref(ms)))
            out[name.value.decode()] = (n.value, ms.value)
        return out

    def last_launch_count(self):
        return lib().df_moe_last_launch_count(self.h)

    def cache_stats(self):
        """(hits, misses, bytes copied host -> HBM) of the expert cache."""
        hits, misses, nbytes = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        self._check(lib().df_moe_cache_stats(self.h, ctypes.byref(hits), ctypes.byref(misses),
                                             ctypes.byref(nbytes)))
        return hits.value, misses.value, nbytes.value

    def graph(self, x, T, out, ids, weights, residual=None, out_f32=None):
        """A forward pass captured into a CUDA graph (df_moe_graph_create),
        bound to these buffers: replay with Graph.launch after changing the
        contents of x."""
        g = ctypes.c_void_p()
        self._check(lib().df_moe_graph_create(self.h, _ptr(x), T, _ptr(residual), _ptr(out),
                                              _ptr(out_f32), _ptr(ids), _ptr(weights),
                                              ctypes.byref(g)))
        return Graph(g)


class Graph:
    """Owns one df_moe_graph."""

    def __init__(self, g):
        self.g = g

    def launch(self, stream=None):
        rc = lib().df_moe_graph_launch(self.g, _stream(stream))
        if rc != OK:
            raise DfMoeError(rc, lib().df_moe_last_error(None).decode())

    def launch_count(self):
        return lib().df_moe_graph_launch_count(self.g)

    def close(self):
        if self.g:
            lib().df_moe_graph_destroy(self.g)
            self.g = None

    def __del__(self):
        self.close()


def stream_read(buf, nbytes, sink, stream=None):
    """Read-only streaming probe over nbytes of device memory (df_moe_stream_read)."""
    rc = lib().df_moe_stream_read(_ptr(buf), nbytes, _ptr(sink), _stream(stream))
    if rc != OK:
        raise DfMoeError(rc, lib().df_moe_last_error(None).decode())
