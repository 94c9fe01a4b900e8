"""The C-ABI library builds, loads, exports every entry point the header
declares, and refuses bad arguments on the host (no GPU needed: every call
here is rejected before anything touches a device)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8d.h")


@pytest.fixture(scope="module")
def q8d():
    from q8_block_quantized_matvec_gb300 import build
    build.build()
    import q8_block_quantized_matvec_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q8d_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("q8d_matvec", "q8d_matmul_small_m", "q8d_matmul_small_m_ws",
                 "q8d_matmul_small_m_workspace_bytes", "q8d_kv_append", "q8d_gqa_decode_attn",
                 "q8d_gqa_workspace_bytes", "q8d_step_create", "q8d_step_launch",
                 "q8d_step_status", "q8d_step_destroy", "q8d_step_launch_host"):
        assert want in names


def test_every_declared_symbol_is_exported(q8d):
    L = q8d.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_strerror_and_version(q8d):
    assert q8d.lib().q8d_version() >= 100
    for s in range(-7, 1):
        assert q8d.strerror(s) != "unknown status"
    assert q8d.strerror(-99) == "unknown status"


A16 = 0x10000  # fake, 16-byte aligned addresses: every call below is refused first
B16 = 0x20000
C16 = 0x30000


def test_matvec_refusals(q8d):
    L = q8d.lib()
    assert L.q8d_matvec(A16, B16, C16, 1000, 4, None) == q8d.Q8D_EUNSUPPORTED   # n % 32
    assert L.q8d_matvec(None, B16, C16, 64, 4, None) == q8d.Q8D_EINVAL
    assert L.q8d_matvec(A16, None, C16, 64, 4, None) == q8d.Q8D_EINVAL
    assert L.q8d_matvec(A16, B16, None, 64, 4, None) == q8d.Q8D_EINVAL
    assert L.q8d_matvec(A16, B16 + 2, C16, 64, 4, None) == q8d.Q8D_EALIGN      # weights
    assert L.q8d_matvec(A16 + 4, B16, C16, 64, 4, None) == q8d.Q8D_EALIGN      # x
    assert L.q8d_matvec(A16, B16, A16 + 8, 64, 4, None) == q8d.Q8D_EINVAL      # out overlaps x
    assert L.q8d_matvec(A16, B16, C16, -32, 4, None) == q8d.Q8D_EINVAL
    assert L.q8d_matvec(A16, B16, C16, 64, 0, None) == q8d.Q8D_OK              # empty: no-op


def test_small_m_refusals(q8d):
    L = q8d.lib()
    assert L.q8d_matmul_small_m(A16, 64, B16, C16, 4, 300, 64, 4, None) == q8d.Q8D_EUNSUPPORTED
    assert L.q8d_matmul_small_m(A16, 32, B16, C16, 4, 2, 64, 4, None) == q8d.Q8D_EINVAL  # ldx < n
    assert L.q8d_matmul_small_m(A16, 64, B16, C16, 3, 2, 64, 4, None) == q8d.Q8D_EINVAL  # ldy < p
    assert L.q8d_matmul_small_m(A16, 66, B16, C16, 4, 2, 64, 4, None) == q8d.Q8D_EALIGN
    assert L.q8d_matmul_small_m(A16, 64, B16, C16, 4, 2, 48, 4, None) == q8d.Q8D_EUNSUPPORTED
    assert L.q8d_matmul_small_m(A16, 64, B16, C16, 4, 0, 64, 4, None) == q8d.Q8D_OK


def test_small_m_workspace_bytes(q8d):
    """2 bytes per element of m rows rounded up to 16 per 128-row block, for
    the shapes the tensor-core path takes (9 <= m <= 256, n % 256 == 0)."""
    W = q8d.q8d_matmul_small_m_workspace_bytes
    scales = lambda m: 16 * ((m + 3) // 4)               # the rows' inverse scales
    assert W(8, 3584) == 0 and W(0, 3584) == 0 and W(257, 512) == 0
    assert W(16, 3600) == 0 and W(16, 96) == 0          # n % 256 != 0: CUDA cores
    assert W(9, 3584) == 2 * 3584 * 16 + scales(9)
    assert W(16, 3584) == 2 * 3584 * 16 + scales(16)
    assert W(64, 18944) == 2 * 18944 * 64 + scales(64)
    assert W(130, 256) == 2 * 256 * (128 + 16) + scales(130)
    assert W(256, 512) == 2 * 512 * 256 + scales(256)


def test_small_m_ws_refusals(q8d):
    L = q8d.lib()
    need = q8d.q8d_matmul_small_m_workspace_bytes(16, 256)
    D16 = 0x40000
    args = (A16, 256, B16, C16, 4, 16, 256, 4)
    assert L.q8d_matmul_small_m_ws(*args, None, need, None) == q8d.Q8D_EINVAL        # needed
    assert L.q8d_matmul_small_m_ws(*args, D16, need - 16, None) == q8d.Q8D_EINVAL    # too small
    assert L.q8d_matmul_small_m_ws(*args, D16 + 8, need, None) == q8d.Q8D_EALIGN
    assert L.q8d_matmul_small_m_ws(*args, A16 + 4096, need, None) == q8d.Q8D_EINVAL  # overlaps X
    assert L.q8d_matmul_small_m_ws(*args, C16 - 64, need, None) == q8d.Q8D_EINVAL   # overlaps Y
    assert L.q8d_matmul_small_m_ws(A16, 32, B16, C16, 4, 16, 256, 4, D16, need, None) == q8d.Q8D_EINVAL
    assert L.q8d_matmul_small_m_ws(A16, 256, B16, C16, 4, 0, 256, 4, None, 0, None) == q8d.Q8D_OK
    assert L.q8d_matmul_small_m_ws(A16, 256, B16, C16, 4, 300, 256, 4, D16, need, None) == \
        q8d.Q8D_EUNSUPPORTED


def test_kv_append_refusals(q8d):
    L = q8d.lib()
    assert L.q8d_kv_append(A16, B16, C16, C16 + 4096, 7, 64, 8, A16, A16, None) == q8d.Q8D_EUNSUPPORTED
    assert L.q8d_kv_append(None, B16, C16, C16 + 4096, 1, 64, 8, A16, A16, None) == q8d.Q8D_EINVAL
    assert L.q8d_kv_append(A16, B16, C16, C16 + 4096, 1, 64, 8, None, A16, None) == q8d.Q8D_EINVAL
    assert L.q8d_kv_append(A16, B16, C16, C16 + 64, 1, 64, 8, A16, A16, None) == q8d.Q8D_EINVAL  # caches overlap
    # packed Q8_0: rows must be whole blocks; caches of cap * kv_width/32 * 34 bytes
    assert L.q8d_kv_append(A16, B16, C16, C16 + 4096, 2, 48, 8, A16, A16, None) == q8d.Q8D_EUNSUPPORTED
    assert L.q8d_kv_append(A16, B16, C16, C16 + 496, 2, 64, 8, A16, A16, None) == q8d.Q8D_EINVAL
    assert L.q8d_kv_append(A16, B16, C16 + 2, C16 + 4096, 2, 64, 8, A16, A16, None) == q8d.Q8D_EALIGN


def attn(q8d, **kw):
    a = dict(q=A16, k_new=None, v_new=None, kc=B16, vc=C16, dt=1, out=A16 + 0x100000, batch=1,
             H=16, Hk=8, D=128, cap=64, stride=0, lens=A16, scale=0.088, ws=A16 + 0x200000,
             wsb=1 << 30, err=A16)
    a.update(kw)
    return q8d.lib().q8d_gqa_decode_attn(a["q"], a["k_new"], a["v_new"], a["kc"], a["vc"], a["dt"],
                                         a["out"], a["batch"], a["H"], a["Hk"], a["D"], a["cap"],
                                         a["stride"], a["lens"], a["scale"], a["ws"], a["wsb"],
                                         a["err"], None)


def test_attention_refusals(q8d):
    assert attn(q8d, D=96) == q8d.Q8D_EUNSUPPORTED
    assert attn(q8d, H=12, Hk=8) == q8d.Q8D_EUNSUPPORTED
    assert attn(q8d, H=64, Hk=2) == q8d.Q8D_EUNSUPPORTED          # group of 32 > 16
    assert attn(q8d, dt=3) == q8d.Q8D_EUNSUPPORTED
    assert attn(q8d, k_new=A16) == q8d.Q8D_EINVAL                 # k without v
    assert attn(q8d, ws=None) == q8d.Q8D_EINVAL
    assert attn(q8d, kc=B16 + 8) == q8d.Q8D_EALIGN
    assert attn(q8d, batch=2, stride=100) == q8d.Q8D_EINVAL        # sequences would overlap
    assert attn(q8d, wsb=16) == q8d.Q8D_ERANGE
    assert attn(q8d, scale=float("inf")) == q8d.Q8D_EINVAL
    # packed cache: sequence starts (stride / 32 * 34 bytes) must be 16-byte aligned
    big = 64 * 1024 * 128
    assert attn(q8d, dt=2, batch=2, stride=big + 32) == q8d.Q8D_EALIGN
    assert attn(q8d, dt=2, batch=2, stride=big + 8) == q8d.Q8D_EALIGN


def test_window_attention_refusals(q8d):
    L = q8d.lib()

    def win(**kw):
        a = dict(runs=A16 + 0x300000, stride=0, batch=2, dt=1, kc=B16)
        a.update(kw)
        return L.q8d_gqa_decode_attn_window(A16, None, None, a["kc"], C16, a["dt"], A16 + 0x100000,
                                            a["batch"], 16, 8, 128, 64, a["stride"], a["runs"],
                                            0.088, A16 + 0x200000, 1 << 30, A16, None)
    assert win(runs=None) == q8d.Q8D_EINVAL
    assert win(stride=100) == q8d.Q8D_EINVAL        # overlapping per-sequence caches
    assert win(runs=A16 + 0x300002) == q8d.Q8D_EALIGN
    assert win(kc=B16 + 8) == q8d.Q8D_EALIGN
    assert win(dt=5) == q8d.Q8D_EUNSUPPORTED


def test_step_create_refusals(q8d):
    L = q8d.lib()
    h = C.c_void_p()
    assert L.q8d_step_create(None, None, C.byref(h)) == q8d.Q8D_EINVAL
    assert L.q8d_step_launch_host(None, None, None, None) == q8d.Q8D_EINVAL
    layers = (q8d.LayerDesc * 1)()
    for nm, _ in q8d.LayerDesc._fields_:
        setattr(layers[0], nm, A16)
    d = q8d.StepDesc(64, 1, 4, 2, 80, 64, 10, 0, 0, 1, 8, 1e-6, 1e6, A16, A16, A16,
                     C.cast(layers, C.POINTER(q8d.LayerDesc)), A16, A16, A16, None)
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EUNSUPPORTED  # head_dim 80
    d.head_dim = 64
    d.n_heads = 3
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EUNSUPPORTED  # H % Hk
    d.n_heads = 26
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EUNSUPPORTED  # 13 > 12, f16
    d.n_heads = 34
    d.kv_dtype = 0
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EUNSUPPORTED  # 17 > 16
    d.kv_dtype = 1
    d.n_heads = 4
    d.embed = A16 + 2
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EALIGN
    d.embed = A16
    d.out_norm = A16 + 4                                  # RMSNorm weights: float4 loads
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EALIGN
    d.out_norm = A16
    layers[0].ffn_norm = A16 + 4
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EALIGN
    layers[0].ffn_norm = A16
    layers[0].bk = A16 + 2                                # element loads need 4 bytes
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EALIGN
    layers[0].bk = A16
    d.qk_norm = 1
    layers[0].q_norm = None
    assert L.q8d_step_create(C.byref(d), None, C.byref(h)) == q8d.Q8D_EINVAL
    assert h.value is None
