"""ctypes front end of the scalar C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and
by bench.py's cpu_baseline / reference leg, never by the product package.
It builds liboracle.so from oracle.c with gcc on first use (or via build()).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

KV_F32 = 0
KV_F16 = 1
KV_Q8_0 = 2  # packed rows of kv_width/32 Q8_0 blocks (34 bytes each)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no fp contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


class Layer(C.Structure):
    _fields_ = [(nm, C.c_void_p) for nm in
                ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "attn_norm", "ffn_norm", "q_norm",
                 "k_norm", "bq", "bk", "bv", "kcache", "vcache")]


class Model(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_layers", C.c_int), ("n_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("qk_norm", C.c_int), ("qkv_bias", C.c_int),
                ("kv_dtype", C.c_int), ("cap", C.c_int), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("embed", C.c_void_p), ("out_norm", C.c_void_p),
                ("lm_head", C.c_void_p), ("layers", C.POINTER(Layer))]


def _declare(L):
    vp, i32, i64, f32 = C.c_void_p, C.c_int, C.c_int64, C.c_float
    L.orc_f16_to_f32.argtypes = [C.c_uint16]
    L.orc_f16_to_f32.restype = f32
    L.orc_f32_to_f16.argtypes = [f32]
    L.orc_f32_to_f16.restype = C.c_uint16
    L.orc_q8_dequant_row.argtypes = [vp, i64, i32, vp]
    L.orc_q8_matvec.argtypes = [vp, vp, i32, i32, vp, vp, i32]
    L.orc_q8_matvec_rows.argtypes = [vp, vp, i32, vp, i32, vp, vp]
    L.orc_q8_matmul.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, i32]
    L.orc_kv_append.argtypes = [vp, vp, vp, vp, i32, i32, i64]
    L.orc_q8_0_quantize_block.argtypes = [vp, vp]
    L.orc_gqa_decode_attn.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp]
    L.orc_gqa_decode_attn.restype = i32
    L.orc_gqa_decode_attn_runs.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, f32, vp,
                                           vp]
    L.orc_gqa_decode_attn_runs.restype = i32
    L.orc_rmsnorm.argtypes = [vp, vp, i32, C.c_double, vp]
    L.orc_rope_head.argtypes = [vp, i32, i64, C.c_double]
    L.orc_silu_mul.argtypes = [C.c_double, C.c_double]
    L.orc_silu_mul.restype = C.c_double
    L.orc_argmax.argtypes = [vp, i64]
    L.orc_argmax.restype = i64
    L.orc_decode_step.argtypes = [C.POINTER(Model), i64, i64, vp, C.POINTER(i64), i32]
    L.orc_decode_step.restype = i32


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------------------
def f16_to_f32(bits: int) -> float:
    return float(lib().orc_f16_to_f32(int(bits) & 0xFFFF))


def f32_to_f16(x) -> int:
    return int(lib().orc_f32_to_f16(float(np.float32(x))))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    f = lib().orc_f32_to_f16
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.fromiter((f(float(v)) for v in flat), dtype=np.uint16, count=flat.size).reshape(x.shape)


def dequant_row(w: np.ndarray, row: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().orc_q8_dequant_row(_p(np.ascontiguousarray(w)), int(row), int(n), _p(out))
    return out


def q8_matvec(w: np.ndarray, x: np.ndarray, n: int, p: int, nthreads: int | None = None):
    """Returns (out f32[p], absterm f64[p])."""
    w = np.ascontiguousarray(w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size >= n and w.size >= p * (n // 32) * 34
    out = np.empty(p, dtype=np.float32)
    ab = np.empty(p, dtype=np.float64)
    lib().orc_q8_matvec(_p(w), _p(x), n, p, _p(out), _p(ab), nthreads or default_threads())
    return out, ab


def q8_matvec_rows(w: np.ndarray, x: np.ndarray, n: int, rows):
    w = np.ascontiguousarray(w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty(rows.size, dtype=np.float32)
    ab = np.empty(rows.size, dtype=np.float64)
    lib().orc_q8_matvec_rows(_p(w), _p(x), n, _p(rows), rows.size, _p(out), _p(ab))
    return out, ab


def q8_matmul(w: np.ndarray, X: np.ndarray, n: int, p: int, nthreads: int | None = None):
    """X [m, n] f32 -> (Y [m, p] f32, absterm [m, p] f64)."""
    w = np.ascontiguousarray(w)
    X = np.ascontiguousarray(X, dtype=np.float32)
    m = X.shape[0]
    Y = np.empty((m, p), dtype=np.float32)
    ab = np.empty((m, p), dtype=np.float64)
    lib().orc_q8_matmul(_p(w), _p(X), X.shape[1], m, n, p, _p(Y), p, _p(ab),
                        nthreads or default_threads())
    return Y, ab


def q8_0_quantize_block(x) -> np.ndarray:
    """The packed-KV store's quantizer on 32 values: 34 bytes (uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 32
    out = np.empty(34, dtype=np.uint8)
    lib().orc_q8_0_quantize_block(_p(x), _p(out))
    return out


def kv_row_bytes(kv_dtype: int, kv_width: int) -> int:
    if kv_dtype == KV_F32:
        return 4 * kv_width
    if kv_dtype == KV_F16:
        return 2 * kv_width
    return kv_width // 32 * 34


def kv_append(k, v, kc: np.ndarray, vc: np.ndarray, kv_dtype: int, pos: int):
    """Writes row `pos` of the host caches in place."""
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert kc.flags.c_contiguous and vc.flags.c_contiguous
    lib().orc_kv_append(_p(k), _p(v), _p(kc), _p(vc), kv_dtype, k.size, int(pos))


def gqa_decode_attn(q, kc, vc, kv_dtype: int, n_heads: int, n_kv_heads: int, head_dim: int,
                    L: int, scale: float):
    """One sequence: q f32[H*d]; caches [cap, Hk*d] (f16 or f32).  Returns
    (out f32[H*d], absterm f64[H*d])."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    kc = np.ascontiguousarray(kc)
    vc = np.ascontiguousarray(vc)
    out = np.empty(n_heads * head_dim, dtype=np.float32)
    ab = np.empty(n_heads * head_dim, dtype=np.float64)
    rc = lib().orc_gqa_decode_attn(_p(q), _p(kc), _p(vc), kv_dtype, n_heads, n_kv_heads, head_dim,
                                   int(L), float(scale), _p(out), _p(ab))
    if rc != 0:
        raise ValueError("oracle attention: bad arguments")
    return out, ab


def gqa_decode_attn_runs(q, kc, vc, kv_dtype: int, n_heads: int, n_kv_heads: int, head_dim: int,
                         runs, scale: float):
    """Windowed attention of one query: the cache rows of `runs` ((cell, len)
    pairs over a cache of kc.shape[0] rows).  Returns (out f32[H*d],
    absterm f64[H*d])."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    kc = np.ascontiguousarray(kc)
    vc = np.ascontiguousarray(vc)
    r = np.ascontiguousarray(np.asarray(runs, dtype=np.int32).reshape(-1, 2))
    out = np.empty(n_heads * head_dim, dtype=np.float32)
    ab = np.empty(n_heads * head_dim, dtype=np.float64)
    rc = lib().orc_gqa_decode_attn_runs(_p(q), _p(kc), _p(vc), kv_dtype, n_heads, n_kv_heads,
                                        head_dim, kc.shape[0], _p(r), r.shape[0], float(scale),
                                        _p(out), _p(ab))
    if rc != 0:
        raise ValueError("oracle windowed attention: bad runs")
    return out, ab


def rmsnorm(x, w, eps):
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), _p(w), x.size, float(eps), _p(out))
    return out


def rope_head(x, pos, theta):
    x = np.array(x, dtype=np.float64)
    lib().orc_rope_head(_p(x), x.size, int(pos), float(theta))
    return x


def silu_mul(g, u) -> float:
    return lib().orc_silu_mul(float(g), float(u))


def argmax(x) -> int:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return int(lib().orc_argmax(_p(x), x.size))


class HostStep:
    """Host-side model for orc_decode_step: keeps the numpy arrays alive and
    owns the oracle's own KV caches."""

    def __init__(self, weights, cap: int, caches=None):
        s = weights.shape
        self.shape = s
        self.w = weights
        self.cap = cap
        dt = np.float16 if s.kv_dtype == KV_F16 else np.float32
        if caches is None:
            caches = [(np.zeros((cap, s.kv_width), dt), np.zeros((cap, s.kv_width), dt))
                      for _ in range(s.n_layers)]
        self.caches = [(np.ascontiguousarray(k), np.ascontiguousarray(v)) for k, v in caches]
        self._layers = (Layer * s.n_layers)()
        for li, L in enumerate(weights.layers):
            lay = self._layers[li]
            for nm in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "attn_norm", "ffn_norm"):
                setattr(lay, nm, L[nm].ctypes.data)
            for nm in ("q_norm", "k_norm", "bq", "bk", "bv"):
                setattr(lay, nm, L[nm].ctypes.data if nm in L else None)
            lay.kcache = self.caches[li][0].ctypes.data
            lay.vcache = self.caches[li][1].ctypes.data
        self.model = Model(s.hidden, s.n_layers, s.n_heads, s.n_kv_heads, s.head_dim, s.ffn,
                           s.vocab, int(s.qk_norm), int(s.qkv_bias), s.kv_dtype, cap,
                           s.rms_eps, s.rope_theta, weights.embed.ctypes.data,
                           weights.out_norm.ctypes.data, weights.lm_head.ctypes.data,
                           self._layers)

    def step(self, token: int, pos: int, nthreads: int | None = None):
        """Runs one decode step in double; appends row `pos` to the oracle's
        caches.  Returns (logits f32[vocab], next_token)."""
        logits = np.empty(self.shape.vocab, dtype=np.float32)
        nxt = C.c_int64(-1)
        rc = lib().orc_decode_step(C.byref(self.model), int(token), int(pos), _p(logits),
                                   C.byref(nxt), nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle decode step: bad token or position")
        return logits, int(nxt.value)
