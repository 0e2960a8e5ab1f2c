"""Python binding of libpopffn.so: partition-guided online structured pruning (POP) of a gated-MLP FFN.

This module only marshals arguments: every step of prefill, partition and decode
runs in the library's sm_103a kernels. PyTorch supplies device memory
(``tensor.data_ptr()``) and streams (``torch.cuda.current_stream().cuda_stream``).
There is no CPU fallback: importing fails loudly when the library is missing.

The names mirror the C ABI in ``include/pop_ffn.h`` (``pop_ffn_create``,
``pop_prefill_partition``, ``pop_decode_step``, ``pop_ffn_dense_ref``, ...);
``PopFFN`` wraps a handle for convenience.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpopffn.so")

POP_OK, POP_ERR_INVALID_ARG, POP_ERR_STATE, POP_ERR_CUDA, POP_ERR_OOM, POP_ERR_TIMEOUT, POP_ERR_UNSUPPORTED, \
    POP_ERR_DEVICE = range(8)
POP_MAX_D, POP_MAX_D_FF, POP_MAX_BATCH, POP_STATIC_MAX_D_FF = 16384, 49152, 64, 49152


class pop_config(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("D_FF", ctypes.c_int), ("r", ctypes.c_double), ("gamma", ctypes.c_double),
                ("period", ctypes.c_int), ("max_batch", ctypes.c_int), ("max_prefill_tokens", ctypes.c_int),
                ("out_f32", ctypes.c_int), ("skip", ctypes.c_int)]


class pop_counts(ctypes.Structure):
    _fields_ = [("n_P", ctypes.c_int), ("n_R", ctypes.c_int), ("n_C", ctypes.c_int), ("keep", ctypes.c_int),
                ("k", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class PopError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


_vp, _i32, _f64, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_uint64
_ip, _fp = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float)
SIGNATURES = {
    "pop_region_counts": (_i32, [_i32, _f64, _f64, ctypes.POINTER(pop_counts)]),
    "pop_ffn_create": (_i32, [ctypes.POINTER(pop_config), _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)]),
    "pop_ffn_destroy": (None, [_vp]),
    "pop_ffn_counts": (_i32, [_vp, ctypes.POINTER(pop_counts)]),
    "pop_prefill_partition": (_i32, [_vp, _vp, _i32, _vp, _vp]),
    "pop_partition_from_importance": (_i32, [_vp, _vp, _vp]),
    "pop_set_partition": (_i32, [_vp, _ip, _ip, _ip, _vp]),
    "pop_decode_step": (_i32, [_vp, _vp, _i32, _vp, _vp]),
    "pop_ffn_dense_ref": (_i32, [_vp, _vp, _i32, _vp, _vp]),
    "pop_get_partition": (_i32, [_vp, _ip, _ip, _ip]),
    "pop_get_importance": (_i32, [_vp, _fp, _fp]),
    "pop_get_selected": (_i32, [_vp, _ip, _ip]),
    "pop_get_scores": (_i32, [_vp, _fp, _fp]),
    "pop_get_step": (_i32, [_vp, _ip]),
    "pop_set_wait_limit": (_i32, [_vp, _u64]),
    "pop_profile_enable": (_i32, [_vp, _i32]),
    "pop_profile_read": (_i32, [_vp, ctypes.POINTER(ctypes.c_double), _ip]),
    "pop_ffn_dense_token_noalloc": (_i32, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp]),
    "pop_check": (_i32, [_vp]),
    "pop_last_error": (ctypes.c_char_p, [_vp]),
    "pop_status_string": (ctypes.c_char_p, [_i32]),
    # MoE layer (include/pop_moe.h)
    "pop_moe_create": (_i32, [ctypes.POINTER(pop_config), _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                              ctypes.POINTER(_vp), _vp, ctypes.POINTER(_vp)]),
    "pop_moe_destroy": (None, [_vp]),
    "pop_moe_prefill_partition": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp]),
    "pop_moe_decode_step": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp]),
    "pop_moe_get_routing": (_i32, [_vp, _ip, _ip, _fp]),
    "pop_moe_get_counts": (_i32, [_vp, _ip]),
    "pop_moe_expert": (_vp, [_vp, _i32]),
    "pop_moe_num_experts": (_i32, [_vp]),
    "pop_moe_check": (_i32, [_vp]),
    "pop_moe_set_concurrent": (_i32, [_vp, _i32]),
    "pop_moe_last_error": (ctypes.c_char_p, [_vp]),
}

_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libpopffn.so and declares its signatures. Raises ImportError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_name(s: int) -> str:
    names = ["POP_OK", "POP_ERR_INVALID_ARG", "POP_ERR_STATE", "POP_ERR_CUDA", "POP_ERR_OOM", "POP_ERR_TIMEOUT",
             "POP_ERR_UNSUPPORTED", "POP_ERR_DEVICE"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


def _check(status: int, handle=None):
    if status != POP_OK:
        msg = load_library().pop_last_error(handle)
        raise PopError(status, msg.decode() if msg else "")


def _check_moe(status: int, handle=None):
    if status != POP_OK:
        msg = load_library().pop_moe_last_error(handle)
        raise PopError(status, msg.decode() if msg else "")


def _ptr(t):
    """Device address of a tensor (or an int already holding one, or None)."""
    if t is None or isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _expect(t, name, dtype, shape, min_rows=0):
    """Checks a tensor argument before its address goes to the C ABI: dtype, contiguity and shape
    (None in `shape` accepts any extent; an output may have more rows than it receives, at least
    `min_rows`). Raises PopError(POP_ERR_INVALID_ARG)."""
    if t is None:
        return
    ok = (t.dtype == dtype and t.is_contiguous() and t.dim() == len(shape)
          and all(want is None or got == want for got, want in zip(t.shape, shape))
          and (t.dim() == 0 or t.shape[0] >= min_rows))
    if not ok:
        raise PopError(POP_ERR_INVALID_ARG, f"{name}: expected a contiguous {dtype} tensor of shape "
                                            f"{tuple('*' if w is None else w for w in shape)}, got "
                                            f"{t.dtype} {tuple(t.shape)}{'' if t.is_contiguous() else ' (strided)'}")


def _int_array(a):
    import numpy as np
    arr = np.ascontiguousarray(a, dtype=np.int32)
    if arr.size == 0:
        arr = np.zeros(1, dtype=np.int32)
    return arr, arr.ctypes.data_as(_ip)


# ------------------------------------------------------------------ C-ABI mirrors

def pop_region_counts(N: int, r: float, gamma: float) -> pop_counts:
    out = pop_counts()
    _check(load_library().pop_region_counts(N, r, gamma, ctypes.byref(out)))
    return out


def pop_ffn_create(cfg: pop_config, Wg, W1, W2, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(load_library().pop_ffn_create(ctypes.byref(cfg), _ptr(Wg), _ptr(W1), _ptr(W2), _stream(stream),
                                         ctypes.byref(h)))
    return h.value


def pop_ffn_destroy(h) -> None:
    load_library().pop_ffn_destroy(h)


def pop_ffn_counts(h) -> pop_counts:
    out = pop_counts()
    _check(load_library().pop_ffn_counts(h, ctypes.byref(out)), h)
    return out


def pop_prefill_partition(h, X, M: int, Y=None, stream=None) -> None:
    _check(load_library().pop_prefill_partition(h, _ptr(X), M, _ptr(Y), _stream(stream)), h)


def pop_partition_from_importance(h, importance, stream=None) -> None:
    _check(load_library().pop_partition_from_importance(h, _ptr(importance), _stream(stream)), h)


def pop_set_partition(h, R, C, P, stream=None) -> None:
    (_r, rp), (_c, cp), (_p, pp) = _int_array(R), _int_array(C), _int_array(P)
    _check(load_library().pop_set_partition(h, rp, cp, pp, _stream(stream)), h)


def pop_decode_step(h, x, B: int, y, stream=None) -> None:
    _check(load_library().pop_decode_step(h, _ptr(x), B, _ptr(y), _stream(stream)), h)


def pop_ffn_dense_ref(h, X, M: int, Y, stream=None) -> None:
    _check(load_library().pop_ffn_dense_ref(h, _ptr(X), M, _ptr(Y), _stream(stream)), h)


def pop_get_partition(h):
    import numpy as np
    c = pop_ffn_counts(h)
    R, C, P = (np.zeros(max(n, 1), dtype=np.int32) for n in (c.n_R, c.n_C, c.n_P))
    _check(load_library().pop_get_partition(h, R.ctypes.data_as(_ip), C.ctypes.data_as(_ip), P.ctypes.data_as(_ip)),
           h)
    return R[:c.n_R], C[:c.n_C], P[:c.n_P]


def pop_get_importance(h):
    import numpy as np
    c = pop_ffn_counts(h)
    N = c.n_P + c.n_R + c.n_C
    I, ss = np.zeros(N, dtype=np.float32), np.zeros(N, dtype=np.float32)
    _check(load_library().pop_get_importance(h, I.ctypes.data_as(_fp), ss.ctypes.data_as(_fp)), h)
    return I, ss


def pop_get_selected(h):
    import numpy as np
    c = pop_ffn_counts(h)
    S = np.zeros(max(c.k, 1), dtype=np.int32)
    k = ctypes.c_int()
    _check(load_library().pop_get_selected(h, ctypes.byref(k), S.ctypes.data_as(_ip)), h)
    return S[:k.value]


def pop_get_scores(h):
    import numpy as np
    c = pop_ffn_counts(h)
    a, m = np.zeros(max(c.n_C, 1), dtype=np.float32), np.zeros(max(c.n_C, 1), dtype=np.float32)
    _check(load_library().pop_get_scores(h, a.ctypes.data_as(_fp), m.ctypes.data_as(_fp)), h)
    return a[:c.n_C], m[:c.n_C]


def pop_get_step(h) -> int:
    s = ctypes.c_int()
    _check(load_library().pop_get_step(h, ctypes.byref(s)), h)
    return s.value


def pop_set_wait_limit(h, ns: int) -> None:
    _check(load_library().pop_set_wait_limit(h, ns), h)


def pop_profile_enable(h, enable: bool = True) -> None:
    _check(load_library().pop_profile_enable(h, 1 if enable else 0), h)


def pop_profile_read(h):
    """(ms per kernel [gate/up, select, down, reduce] summed since the last read, decode steps)."""
    ms = (ctypes.c_double * 4)()
    steps = ctypes.c_int()
    _check(load_library().pop_profile_read(h, ms, ctypes.byref(steps)), h)
    return list(ms), steps.value


def pop_check(h) -> None:
    _check(load_library().pop_check(h), h)


# ------------------------------------------------------------------ convenience wrapper

class PopFFN:
    """One gated-MLP layer with POP pruning, backed by a pop_ffn handle.

    Wg, W1: torch bf16 [D_FF, D] on the current CUDA device; W2: bf16 [D, D_FF].
    """

    def __init__(self, Wg, W1, W2, r: float, gamma: float = 0.1, period: int = 1, max_batch: int = 1,
                 max_prefill_tokens: int = 2048, out_f32: bool = True, skip: bool = False, stream=None):
        N, D = Wg.shape
        self.handle = None
        self.cfg = pop_config(D=D, D_FF=N, r=r, gamma=gamma, period=period, max_batch=max_batch,
                              max_prefill_tokens=max_prefill_tokens, out_f32=1 if out_f32 else 0,
                              skip=1 if skip else 0)
        self.D, self.N = D, N
        self.handle = pop_ffn_create(self.cfg, Wg, W1, W2, stream)
        self.counts = pop_ffn_counts(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            if not getattr(self, "_borrowed", False):
                pop_ffn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def out_dtype(self):
        import torch
        return torch.float32 if self.cfg.out_f32 else torch.bfloat16

    def prefill_partition(self, X, Y=None, stream=None):
        import torch
        _expect(X, "X", torch.bfloat16, (None, self.D))
        _expect(Y, "Y", self.out_dtype(), (None, self.D), X.shape[0])
        pop_prefill_partition(self.handle, X, X.shape[0], Y, stream)

    def partition_from_importance(self, importance, stream=None):
        import torch
        _expect(importance, "importance", torch.float32, (self.N,))
        pop_partition_from_importance(self.handle, importance, stream)

    def set_partition(self, R, C, P, stream=None):
        pop_set_partition(self.handle, R, C, P, stream)

    def decode_step(self, x, y=None, stream=None):
        import torch
        _expect(x, "x", torch.bfloat16, (None, self.D))
        if y is None:
            y = torch.empty((x.shape[0], self.D), dtype=self.out_dtype(), device=x.device)
        _expect(y, "y", self.out_dtype(), (None, self.D), x.shape[0])
        pop_decode_step(self.handle, x, x.shape[0], y, stream)
        return y

    def dense_ref(self, X, Y=None, stream=None):
        import torch
        _expect(X, "X", torch.bfloat16, (None, self.D))
        if Y is None:
            Y = torch.empty((X.shape[0], self.D), dtype=self.out_dtype(), device=X.device)
        _expect(Y, "Y", self.out_dtype(), (None, self.D), X.shape[0])
        pop_ffn_dense_ref(self.handle, X, X.shape[0], Y, stream)
        return Y

    def partition(self):
        return pop_get_partition(self.handle)

    def importance(self):
        return pop_get_importance(self.handle)

    def selected(self):
        return pop_get_selected(self.handle)

    def scores(self):
        return pop_get_scores(self.handle)

    def step_count(self):
        return pop_get_step(self.handle)

    def set_wait_limit(self, ns: int):
        pop_set_wait_limit(self.handle, ns)

    def profile(self, enable: bool = True):
        pop_profile_enable(self.handle, enable)

    def profile_read(self):
        return pop_profile_read(self.handle)

    def check(self):
        pop_check(self.handle)

    @classmethod
    def _borrow(cls, handle, cfg):
        """A view of a layer handle owned elsewhere (an MoE expert): close() leaves it alone."""
        v = cls.__new__(cls)
        v.cfg, v.D, v.N, v.handle, v._borrowed = cfg, cfg.D, cfg.D_FF, handle, True
        v.counts = pop_ffn_counts(handle)
        return v


# ------------------------------------------------------------------ MoE layer

def pop_moe_create(cfg: pop_config, Wg, W1, W2, stream=None) -> int:
    E = len(Wg)
    arr = [(_vp * E)(*[_ptr(w) for w in ws]) for ws in (Wg, W1, W2)]
    out = _vp()
    _check_moe(load_library().pop_moe_create(ctypes.byref(cfg), E, arr[0], arr[1], arr[2], _stream(stream),
                                             ctypes.byref(out)))
    return out.value


class PopMoE:
    """An MoE layer of POP-pruned gated-MLP experts (top-2 routing), backed by a pop_moe handle.

    Wg, W1: lists of torch bf16 [D_FF, D] (one per expert); W2: list of bf16 [D, D_FF].
    """

    def __init__(self, Wg, W1, W2, r: float, gamma: float = 0.1, period: int = 1, max_batch: int = 1,
                 max_prefill_tokens: int = 2048, out_f32: bool = True, stream=None):
        N, D = Wg[0].shape
        self.handle = None
        self.cfg = pop_config(D=D, D_FF=N, r=r, gamma=gamma, period=period, max_batch=max_batch,
                              max_prefill_tokens=max_prefill_tokens, out_f32=1 if out_f32 else 0)
        self.D, self.N, self.E = D, N, len(Wg)
        self.handle = pop_moe_create(self.cfg, Wg, W1, W2, stream)
        self.experts = [PopFFN._borrow(load_library().pop_moe_expert(self.handle, e), self.cfg)
                        for e in range(self.E)]
        self.counts = self.experts[0].counts

    def close(self):
        if getattr(self, "handle", None):
            self.experts = []
            load_library().pop_moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def out_dtype(self):
        import torch
        return torch.float32 if self.cfg.out_f32 else torch.bfloat16

    def prefill_partition(self, X, logits, Y=None, stream=None):
        """X: bf16 [M, D]; logits: float32 [M, E]; Y (optional): [M, D] of out_dtype()."""
        import torch
        _expect(X, "X", torch.bfloat16, (None, self.D))
        _expect(logits, "logits", torch.float32, (None, self.E), X.shape[0])
        _expect(Y, "Y", self.out_dtype(), (None, self.D), X.shape[0])
        _check_moe(load_library().pop_moe_prefill_partition(self.handle, _ptr(X), _ptr(logits), X.shape[0], _ptr(Y),
                                                            _stream(stream)), self.handle)

    def decode_step(self, x, logits, y=None, stream=None):
        import torch
        _expect(x, "x", torch.bfloat16, (None, self.D))
        _expect(logits, "logits", torch.float32, (None, self.E), x.shape[0])
        if y is None:
            y = torch.empty((x.shape[0], self.D), dtype=self.out_dtype(), device=x.device)
        _expect(y, "y", self.out_dtype(), (None, self.D), x.shape[0])
        _check_moe(load_library().pop_moe_decode_step(self.handle, _ptr(x), _ptr(logits), x.shape[0], _ptr(y),
                                                      _stream(stream)), self.handle)
        return y

    def routing(self):
        """(experts [T, 2] int32, weights [T, 2] float32) of the last call. Syncs."""
        import numpy as np
        lib = load_library()
        T = ctypes.c_int(0)
        _check_moe(lib.pop_moe_get_routing(self.handle, ctypes.byref(T), None, None), self.handle)
        ex = np.zeros((max(T.value, 1), 2), dtype=np.int32)
        w = np.zeros((max(T.value, 1), 2), dtype=np.float32)
        _check_moe(lib.pop_moe_get_routing(self.handle, ctypes.byref(T), ex.ctypes.data_as(_ip),
                                           w.ctypes.data_as(_fp)), self.handle)
        return ex[:T.value], w[:T.value]

    def token_counts(self):
        import numpy as np
        c = np.zeros(self.E, dtype=np.int32)
        _check_moe(load_library().pop_moe_get_counts(self.handle, c.ctypes.data_as(_ip)), self.handle)
        return c

    def check(self):
        _check_moe(load_library().pop_moe_check(self.handle), self.handle)

    def set_concurrent(self, on: bool):
        """Experts' decode kernels on streams of their own (True, the default) or one after another
        on the caller's stream (False: for per-kernel timing)."""
        _check_moe(load_library().pop_moe_set_concurrent(self.handle, 1 if on else 0), self.handle)


load_library()
