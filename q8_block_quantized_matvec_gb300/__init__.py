"""Python binding of libq8d, the GB300 Q8_0 decode hot path.

Argument marshalling only: every computation runs in the CUDA kernels of
libq8d.so (built in-tree by build.py for sm_103a).  Functions carry the C
entry points' names and arguments; tensors are torch tensors on the CUDA
device (or raw integer device addresses), `stream` defaults to torch's
current stream.  A non-zero status raises Q8DError.  If the library is
missing the import of any entry point fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libq8d.so")

Q8D_OK = 0
Q8D_EINVAL = -1
Q8D_EALIGN = -2
Q8D_EUNSUPPORTED = -3
Q8D_ERANGE = -4
Q8D_ECUDA = -5
Q8D_ETIMEOUT = -6
Q8D_ENOMEM = -7

Q8D_KV_F32 = 0
Q8D_KV_F16 = 1
Q8D_KV_Q8_0 = 2

Q8D_MAX_RUNS = 4

Q8D_DERR_POS_RANGE = 0x1
Q8D_DERR_LEN_RANGE = 0x2
Q8D_DERR_TOKEN_RANGE = 0x4
Q8D_DERR_WAIT = 0x8


class Q8DError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status}, cuda {last_cuda_error()})")


class LayerDesc(C.Structure):
    _fields_ = [(nm, C.c_void_p) for nm in
                ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "attn_norm", "ffn_norm", "q_norm",
                 "k_norm", "bq", "bk", "bv", "kcache", "vcache")]


class StepDesc(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_layers", C.c_int), ("n_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("qk_norm", C.c_int), ("qkv_bias", C.c_int),
                ("kv_dtype", C.c_int), ("cap", C.c_int), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("embed", C.c_void_p), ("out_norm", C.c_void_p),
                ("lm_head", C.c_void_p), ("layers", C.POINTER(LayerDesc)),
                ("d_token", C.c_void_p), ("d_pos", C.c_void_p), ("d_err", C.c_void_p),
                ("d_logits", C.c_void_p)]


_lib = None


def lib():
    """The loaded libq8d (ctypes CDLL) with argument types declared."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libq8d.so is not built ({LIB_PATH}); run "
                              "q8_block_quantized_matvec_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = C.c_void_p, C.c_int, C.c_longlong, C.c_float, C.c_size_t
        L.q8d_version.restype = i32
        L.q8d_strerror.argtypes = [i32]
        L.q8d_strerror.restype = C.c_char_p
        L.q8d_last_cuda_error.restype = i32
        L.q8d_matvec.argtypes = [vp, vp, vp, i32, i32, vp]
        L.q8d_matvec.restype = i32
        L.q8d_matmul_small_m.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, vp]
        L.q8d_matmul_small_m.restype = i32
        L.q8d_matmul_small_m_workspace_bytes.argtypes = [i32, i32]
        L.q8d_matmul_small_m_workspace_bytes.restype = sz
        L.q8d_matmul_small_m_ws.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, vp, sz, vp]
        L.q8d_matmul_small_m_ws.restype = i32
        L.q8d_kv_append.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.q8d_kv_append.restype = i32
        L.q8d_gqa_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.q8d_gqa_workspace_bytes.restype = sz
        L.q8d_gqa_decode_attn.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                          i64, vp, f32, vp, sz, vp, vp]
        L.q8d_gqa_decode_attn.restype = i32
        L.q8d_gqa_decode_attn_window.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                 i32, i64, vp, f32, vp, sz, vp, vp]
        L.q8d_gqa_decode_attn_window.restype = i32
        L.q8d_noalloc_scratch_bytes.argtypes = []
        L.q8d_noalloc_scratch_bytes.restype = sz
        L.q8d_gqa_decode_attn_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                  i32, i64, vp, f32, vp, vp]
        L.q8d_gqa_decode_attn_noalloc.restype = i32
        L.q8d_step_create.argtypes = [C.POINTER(StepDesc), vp, C.POINTER(vp)]
        L.q8d_step_create.restype = i32
        L.q8d_step_launch.argtypes = [vp, vp]
        L.q8d_step_launch.restype = i32
        L.q8d_step_launch_host.argtypes = [vp, vp, vp, vp]
        L.q8d_step_launch_host.restype = i32
        L.q8d_step_status.argtypes = [vp, vp, i32, C.POINTER(i32)]
        L.q8d_step_status.restype = i32
        L.q8d_step_set_wait_limit.argtypes = [vp, C.c_uint, vp]
        L.q8d_step_set_wait_limit.restype = i32
        L.q8d_step_kernel_count.argtypes = [vp]
        L.q8d_step_kernel_count.restype = i32
        L.q8d_step_logits.argtypes = [vp]
        L.q8d_step_logits.restype = vp
        L.q8d_step_destroy.argtypes = [vp]
        L.q8d_step_destroy.restype = None
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().q8d_strerror(int(status)).decode()


def last_cuda_error() -> int:
    return lib().q8d_last_cuda_error()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> int:
    if status != Q8D_OK:
        raise Q8DError(status, what)
    return status


# ---- entry points (same names and argument order as include/q8d.h) --------

def q8d_matvec(x, w_q8, out, n: int, p: int, stream=None) -> int:
    return _check(lib().q8d_matvec(_ptr(x), _ptr(w_q8), _ptr(out), int(n), int(p),
                                   _stream(stream)), "q8d_matvec")


def q8d_matmul_small_m(X, ldx: int, w_q8, Y, ldy: int, m: int, n: int, p: int, stream=None) -> int:
    return _check(lib().q8d_matmul_small_m(_ptr(X), int(ldx), _ptr(w_q8), _ptr(Y), int(ldy), int(m),
                                           int(n), int(p), _stream(stream)), "q8d_matmul_small_m")


def q8d_matmul_small_m_workspace_bytes(m: int, n: int) -> int:
    return int(lib().q8d_matmul_small_m_workspace_bytes(int(m), int(n)))


def q8d_matmul_small_m_ws(X, ldx: int, w_q8, Y, ldy: int, m: int, n: int, p: int, workspace,
                          ws_bytes: int, stream=None) -> int:
    return _check(lib().q8d_matmul_small_m_ws(_ptr(X), int(ldx), _ptr(w_q8), _ptr(Y), int(ldy),
                                              int(m), int(n), int(p), _ptr(workspace),
                                              int(ws_bytes), _stream(stream)),
                  "q8d_matmul_small_m_ws")


def q8d_kv_append(k, v, kcache, vcache, kv_dtype: int, kv_width: int, cap: int, d_pos, d_err,
                  stream=None) -> int:
    return _check(lib().q8d_kv_append(_ptr(k), _ptr(v), _ptr(kcache), _ptr(vcache), int(kv_dtype),
                                      int(kv_width), int(cap), _ptr(d_pos), _ptr(d_err),
                                      _stream(stream)), "q8d_kv_append")


def q8d_gqa_workspace_bytes(batch: int, n_heads: int, n_kv_heads: int, head_dim: int,
                            max_len: int) -> int:
    return int(lib().q8d_gqa_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, max_len))


def q8d_gqa_decode_attn(q, k_new, v_new, kcache, vcache, kv_dtype: int, out, batch: int,
                        n_heads: int, n_kv_heads: int, head_dim: int, cap: int,
                        cache_batch_stride: int, d_lens, scale: float, workspace, ws_bytes: int,
                        d_err, stream=None) -> int:
    return _check(lib().q8d_gqa_decode_attn(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache), int(kv_dtype), _ptr(out),
        int(batch), int(n_heads), int(n_kv_heads), int(head_dim), int(cap),
        int(cache_batch_stride), _ptr(d_lens), float(scale), _ptr(workspace), int(ws_bytes),
        _ptr(d_err), _stream(stream)), "q8d_gqa_decode_attn")


def q8d_gqa_decode_attn_window(q, k_new, v_new, kcache, vcache, kv_dtype: int, out, batch: int,
                               n_heads: int, n_kv_heads: int, head_dim: int, cap: int,
                               cache_batch_stride: int, d_runs, scale: float, workspace,
                               ws_bytes: int, d_err, stream=None) -> int:
    return _check(lib().q8d_gqa_decode_attn_window(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache), int(kv_dtype), _ptr(out),
        int(batch), int(n_heads), int(n_kv_heads), int(head_dim), int(cap),
        int(cache_batch_stride), _ptr(d_runs), float(scale), _ptr(workspace), int(ws_bytes),
        _ptr(d_err), _stream(stream)), "q8d_gqa_decode_attn_window")


def q8d_noalloc_scratch_bytes() -> int:
    return int(lib().q8d_noalloc_scratch_bytes())


def q8d_gqa_decode_attn_noalloc(q, k_new, v_new, kcache, vcache, kv_dtype: int, out, batch: int,
                                n_heads: int, n_kv_heads: int, head_dim: int, cap: int,
                                cache_batch_stride: int, d_lens, scale: float, d_err,
                                stream=None) -> int:
    """q8d_gqa_decode_attn with the scratch in the library's fixed device
    array (for callers that cannot allocate device memory)."""
    return _check(lib().q8d_gqa_decode_attn_noalloc(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache), int(kv_dtype), _ptr(out),
        int(batch), int(n_heads), int(n_kv_heads), int(head_dim), int(cap),
        int(cache_batch_stride), _ptr(d_lens), float(scale), _ptr(d_err), _stream(stream)),
        "q8d_gqa_decode_attn_noalloc")


class Step:
    """Owns a q8d_step (the captured decode-step graph)."""

    def __init__(self, desc: StepDesc, layers, stream=None):
        self._desc = desc
        self._layers = layers  # keep the ctypes array alive
        h = C.c_void_p()
        _check(lib().q8d_step_create(C.byref(desc), _stream(stream), C.byref(h)), "q8d_step_create")
        self.handle = h.value

    def launch(self, stream=None) -> int:
        return _check(lib().q8d_step_launch(self.handle, _stream(stream)), "q8d_step_launch")

    def launch_host(self, h_token_pos, h_next_token, stream=None) -> int:
        """q8d_step_launch_host: host int32 [token, position] in (or None),
        the next token id out to host int32 [1] (or None); both pinned CPU
        tensors, read the output after synchronising the stream."""
        return _check(lib().q8d_step_launch_host(self.handle, _ptr(h_token_pos), _ptr(h_next_token),
                                                 _stream(stream)), "q8d_step_launch_host")

    def status(self, stream=None, timeout_ms: int = 10000) -> int:
        err = C.c_int(0)
        _check(lib().q8d_step_status(self.handle, _stream(stream), int(timeout_ms), C.byref(err)),
               "q8d_step_status")
        return err.value

    def set_wait_limit(self, polls: int, stream=None) -> int:
        return _check(lib().q8d_step_set_wait_limit(self.handle, int(polls), _stream(stream)),
                      "q8d_step_set_wait_limit")

    def kernel_count(self) -> int:
        return lib().q8d_step_kernel_count(self.handle)

    def logits_ptr(self) -> int:
        return lib().q8d_step_logits(self.handle)

    def close(self):
        if self.handle:
            lib().q8d_step_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q8d_step_create(desc: StepDesc, layers, stream=None) -> Step:
    return Step(desc, layers, stream)
