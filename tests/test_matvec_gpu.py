"""q8d_matvec and q8d_matmul_small_m (CUDA, through the C ABI) against the
oracle.  Bar: |gpu - oracle| <= 1e-5 * sum|terms| per output (f32 path),
2e-3 * sum|terms| for the f16 tensor-core path (m >= 9); exact where the
result is an exact integer or a single product."""
import numpy as np
import pytest
import torch

import synth
from conftest import dev

pytestmark = pytest.mark.gpu

TOL = 1e-5
# the tensor-core path (m >= 9): weights and activations each rounded once
# to f16 (<= 2^-11 relative each), f32 accumulation: ~2^-10 per product
TOL_TC = 2e-3


def gpu_matvec(q8d, w, x, n, p, canary=True):
    wd, xd = dev(w), dev(x)
    pad = 64
    buf = torch.full((p + 2 * pad,), float("nan"), device="cuda")
    out = buf[pad:pad + p]
    q8d.q8d_matvec(xd, wd, out, n, p)
    torch.cuda.synchronize()
    if canary:
        assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + p:]).all(), "wrote outside out"
    return out.cpu().numpy()


SHAPES = [(32, 1), (64, 3), (96, 50), (896, 33), (896, 137), (1024, 3072), (1024, 1),
          (2048, 101), (3072, 77), (3584, 300), (4864, 200), (18944, 67), (160, 999),
          # a few rows per CTA (one tile sized to them): 3, 4 and 5 rows of 20,
          # 2 and 10 column-segment warps
          (18944, 456), (2048, 600), (4864, 750)]


@pytest.mark.parametrize("n,p", SHAPES)
def test_matvec_parity(q8d, orc, n, p):
    w = synth.q8_matrix(0, f"w{n}x{p}", p, n)
    x = synth.normal_f32(0, f"x{n}", n)
    ref, ab = orc.q8_matvec(w, x, n, p)
    got = gpu_matvec(q8d, w, x, n, p)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= TOL * ab), (err / ab).max()


def test_matvec_config0_deterministic(q8d, orc):
    n, p = 1024, 3072
    w = synth.q8_matrix(0, "config0.w", p, n)
    x = synth.normal_f32(0, "config0.x", n)
    a = gpu_matvec(q8d, w, x, n, p)
    b = gpu_matvec(q8d, w, x, n, p)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    ref, ab = orc.q8_matvec(w, x, n, p)
    assert np.all(np.abs(a - ref) <= TOL * ab)


@pytest.mark.parametrize("n,p", [(32, 5), (3584, 64), (18944, 9), (896, 31)])
def test_matvec_exact_integer_sums(q8d, n, p):
    w = synth.q8_from_parts(5, "w", p, n, 0x3C00)
    q = w.reshape(p, n // 32, 34)[:, :, 2:].view(np.int8).astype(np.int64).reshape(p, n)
    got = gpu_matvec(q8d, w, np.ones(n, np.float32), n, p)
    assert np.array_equal(got.astype(np.int64), q.sum(axis=1))


def test_matvec_sum_of_x(q8d):
    n, p = 3584, 5
    w = synth.q8_const_matrix(p, n, 0x3C00, 1)
    x = synth.normal_f32(1, "x", n)
    got = gpu_matvec(q8d, w, x, n, p)
    assert np.all(np.abs(got - np.sum(x, dtype=np.float64)) <= TOL * np.abs(x).sum())


def test_matvec_one_hot(q8d):
    n, p = 128, 7
    w = synth.q8_matrix(9, "w", p, n)
    blk = w.reshape(p, n // 32, 34)
    sc = blk[:, :, 0:2].copy().view("<f2").astype(np.float32).reshape(p, n // 32)
    q = blk[:, :, 2:].view(np.int8).astype(np.float32).reshape(p, n)
    for j in range(n):
        x = np.zeros(n, np.float32)
        x[j] = 1.0
        assert np.array_equal(gpu_matvec(q8d, w, x, n, p, canary=False), sc[:, j // 32] * q[:, j]), j


def test_matvec_minus_128(q8d):
    n, p = 64, 3
    w = synth.q8_const_matrix(p, n, 0x3C00, -128)
    assert np.array_equal(gpu_matvec(q8d, w, np.ones(n, np.float32), n, p), np.full(p, -8192.0, np.float32))


def test_matvec_empty(q8d):
    out = torch.full((5,), 3.0, device="cuda")
    q8d.q8d_matvec(torch.zeros(4, device="cuda"), torch.zeros(16, dtype=torch.uint8, device="cuda"),
                   out, 0, 5)
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros(5, device="cuda"))
    q8d.q8d_matvec(None, None, out, 64, 0)  # p == 0: nothing


def test_matvec_control_perturbed_byte(q8d):
    """A changed weight byte must change exactly its row (guards a vacuous gate)."""
    n, p = 256, 9
    w = synth.q8_matrix(3, "w", p, n)
    x = synth.normal_f32(3, "x", n)
    a = gpu_matvec(q8d, w, x, n, p)
    w2 = w.copy()
    w2[4, 34 * 3 + 7] ^= 0x11
    b = gpu_matvec(q8d, w2, x, n, p)
    assert a[4] != b[4] and np.array_equal(np.delete(a, 4), np.delete(b, 4))


SEVEN_B = [("q/o", 3584, 3584), ("k/v", 3584, 512), ("gate/up", 3584, 18944), ("down", 18944, 3584),
           ("lm_head", 3584, 152064)]


@pytest.mark.parametrize("name,n,p", SEVEN_B)
def test_matvec_7b_shapes_sampled(q8d, orc, name, n, p):
    """Full 7B-shaped matrices, the launch the bench times; 257 sampled rows
    (first, last, seeded random) checked against the oracle row by row."""
    w = synth.q8_matrix(0, f"7b.{name}", p, n)
    x = synth.normal_f32(0, f"7b.x{n}", n)
    got = gpu_matvec(q8d, w, x, n, p)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, p - 1], rng.integers(0, p, 255)])).astype(np.int64)
    ref, ab = orc.q8_matvec_rows(w, x, n, rows)
    assert np.all(np.abs(got[rows] - ref) <= TOL * ab)
    assert np.isfinite(got).all()


# ---------------------------------------------------------------------------- small M
def gpu_small_m(q8d, w, X, n, p, ldx=None, ldy=None):
    m = X.shape[0]
    ldx = ldx or n
    ldy = ldy or p
    Xp = np.zeros((m, ldx), np.float32)
    Xp[:, :n] = X
    Y = torch.full((m, ldy), float("nan"), device="cuda")
    q8d.q8d_matmul_small_m(dev(Xp), ldx, dev(w), Y, ldy, m, n, p)
    torch.cuda.synchronize()
    Yh = Y.cpu().numpy()
    if ldy > p:
        assert np.isnan(Yh[:, p:]).all()
    return Yh[:, :p]


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("n,p", [(3584, 512), (96, 50), (18944, 40), (896, 33)])
def test_small_m_f32_parity(q8d, orc, m, n, p):
    w = synth.q8_matrix(2, f"sm.w{n}", p, n)
    X = synth.normal_f32(2, f"sm.X{n}.{m}", (m, n))
    ref, ab = orc.q8_matmul(w, X, n, p)
    got = gpu_small_m(q8d, w, X, n, p, ldx=n + 4 * (m % 2), ldy=p + 3)
    assert np.all(np.abs(got - ref) <= TOL * ab)


@pytest.mark.parametrize("m", [2, 3, 4, 5, 8])
def test_small_m_matvec_rows_tensor(q8d, orc, m):
    """2 <= m <= 8 on the tensor-core matvec (up to four activation rows per
    launch sharing each decoded weight block; m > 4 in two launches): the
    f32 bar, a ragged row count and padded strides."""
    n, p = 2048, 2500
    w = synth.q8_matrix(13, f"mr.w{n}", p, n)
    X = synth.normal_f32(13, f"mr.X{n}.{m}", (m, n))
    ref, ab = orc.q8_matmul(w, X, n, p)
    got = gpu_small_m(q8d, w, X, n, p, ldx=n + 4, ldy=p + 3)
    assert np.all(np.abs(got - ref) <= TOL * ab)


@pytest.mark.parametrize("m", [9, 16, 64])
@pytest.mark.parametrize("n,p", [(3584, 512), (256, 384), (18944, 128)])
def test_small_m_tensor_parity(q8d, orc, m, n, p):
    w = synth.q8_matrix(4, f"tc.w{n}", p, n)
    X = synth.normal_f32(4, f"tc.X{n}.{m}", (m, n))
    ref, ab = orc.q8_matmul(w, X, n, p)
    got = gpu_small_m(q8d, w, X, n, p)
    assert np.all(np.abs(got - ref) <= TOL_TC * ab)
    # the norm-wise error is reported, and is far inside the bar
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 2e-3


@pytest.mark.parametrize("m", [16, 64])
@pytest.mark.parametrize("n,p", [(3584, 33), (3584, 200), (512, 300)])
def test_small_m_tensor_ragged_row_tile(q8d, orc, m, n, p):
    """p not a multiple of the 128-row tile: the last tile's rows past p come
    from the tensor map's zero fill and are not stored."""
    w = synth.q8_matrix(6, f"tr.w{n}.{p}", p, n)
    X = synth.normal_f32(6, f"tr.X{n}.{m}", (m, n))
    ref, ab = orc.q8_matmul(w, X, n, p)
    got = gpu_small_m(q8d, w, X, n, p, ldy=p + 5)
    assert np.all(np.abs(got - ref) <= TOL_TC * ab)


@pytest.mark.parametrize("p", [300, 10000])  # 3 row tiles: K split in clusters; 79: none
def test_small_m_tensor_scale_range(q8d, orc, p):
    """A block scale above 511.75 (scale * q beyond f16): the outputs of its
    128-row tile are NaN, every other tile is within the bar."""
    m, n = 16, 512
    w = synth.q8_matrix(14, f"rg.w{p}", p, n).copy()
    row, blk = 130, 3  # second row tile
    w[row, blk * 34:blk * 34 + 2] = np.frombuffer(np.float16(1000.0).tobytes(), np.uint8)
    X = synth.normal_f32(14, f"rg.X{n}", (m, n))
    got = gpu_small_m(q8d, w, X, n, p)
    assert np.isnan(got[:, 128:256]).all()
    ref, ab = orc.q8_matmul(w, X, n, p)
    keep = np.r_[0:128, 256:p]
    assert np.all(np.abs(got[:, keep] - ref[:, keep]) <= TOL_TC * ab[:, keep])


@pytest.mark.parametrize("m", [65, 80, 128, 129, 200, 256])
def test_small_m_tensor_large_m(q8d, orc, m):
    """m up to the entry point's 256: above 128 rows the activations go
    through the kernel in more than one pass."""
    n, p = 1024, 300
    w = synth.q8_matrix(7, "lm.w", p, n)
    X = synth.normal_f32(7, f"lm.X{m}", (m, n))
    ref, ab = orc.q8_matmul(w, X, n, p)
    got = gpu_small_m(q8d, w, X, n, p)
    assert np.all(np.abs(got - ref) <= TOL_TC * ab)


@pytest.mark.parametrize("m", [16, 130])
def test_small_m_caller_workspace(q8d, orc, m):
    """q8d_matmul_small_m_ws: one caller workspace serves two calls with
    different activations, and nothing is written outside it."""
    n, p = 512, 300
    w = synth.q8_matrix(9, "ws.w", p, n)
    need = q8d.q8d_matmul_small_m_workspace_bytes(m, n)
    assert need == 2 * n * (m // 128 * 128 + (m % 128 + 15) // 16 * 16) + 16 * ((m + 3) // 4)
    pad = 4096
    buf = torch.full((need + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = buf[pad:pad + need]
    for seed in (10, 11):
        X = synth.normal_f32(seed, f"ws.X{m}", (m, n))
        ref, ab = orc.q8_matmul(w, X, n, p)
        Y = torch.full((m, p), float("nan"), device="cuda")
        q8d.q8d_matmul_small_m_ws(dev(X), n, dev(w), Y, p, m, n, p, ws, need)
        torch.cuda.synchronize()
        assert np.all(np.abs(Y.cpu().numpy() - ref) <= TOL_TC * ab), seed
    assert (buf[:pad] == 0xA5).all() and (buf[pad + need:] == 0xA5).all()


@pytest.mark.parametrize("m", [1, 4, 16, 64])
def test_small_m_bench_shape_sampled(q8d, orc, m):
    """The launch the bench times: 7B gate/up (3584 -> 18944) at m rows;
    257 sampled output rows per activation row against the oracle."""
    n, p = 3584, 18944
    w = synth.q8_matrix(0, "7b.gate/up", p, n)
    X = synth.normal_f32(8, f"bs.X{m}", (m, n))
    got = gpu_small_m(q8d, w, X, n, p)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, p - 1], rng.integers(0, p, 255)])).astype(np.int64)
    tol = TOL if m <= 8 else TOL_TC
    for i in range(m):
        ref, ab = orc.q8_matvec_rows(w, X[i], n, rows)
        assert np.all(np.abs(got[i, rows] - ref) <= tol * ab), i
    assert np.isfinite(got).all()


# ---------------------------------------------------------------------------- tensor-core matvec
# q8d_matvec runs its tensor-core kernel (mma.sync, f16 hi/lo activations)
# for one matrix with n % 256 == 0, n >= 2048 and p >= 16 * SMs rows; these shapes
# reach it (and its sliced-row path for n > 4352), including row counts
# that are not multiples of the 8-row unit.
MMA_SHAPES = [(2048, 3072), (3584, 3584), (3584, 2437), (18944, 3584), (4864, 2500), (2048, 5000),
              (8192, 3001)]


@pytest.mark.parametrize("n,p", MMA_SHAPES)
def test_matvec_mma_parity(q8d, orc, n, p):
    w = synth.q8_matrix(11, f"mm.w{n}x{p}", p, n)
    x = synth.normal_f32(11, f"mm.x{n}", n)
    ref, ab = orc.q8_matvec(w, x, n, p)
    got = gpu_matvec(q8d, w, x, n, p)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= TOL * ab), (err / ab).max()


@pytest.mark.parametrize("n,p", [(2048, 2500), (3584, 2440), (18944, 2432)])
def test_matvec_mma_exact_integer_sums(q8d, n, p):
    w = synth.q8_from_parts(5, "mmw", p, n, 0x3C00)
    q = w.reshape(p, n // 32, 34)[:, :, 2:].view(np.int8).astype(np.int64).reshape(p, n)
    got = gpu_matvec(q8d, w, np.ones(n, np.float32), n, p)
    assert np.array_equal(got.astype(np.int64), q.sum(axis=1))


def test_matvec_mma_one_hot_columns(q8d):
    """One-hot x at columns covering every byte position of even and odd
    blocks (the permuted word order of both alignments)."""
    n, p = 2048, 2432
    w = synth.q8_matrix(12, "mmoh", p, n)
    blk = w.reshape(p, n // 32, 34)
    sc = blk[:, :, 0:2].copy().view("<f2").astype(np.float32).reshape(p, n // 32)
    q = blk[:, :, 2:].view(np.int8).astype(np.float32).reshape(p, n)
    for j in list(range(0, 64)) + [97, 130, 255, 256, 319, 480, 511, 1024, 2047]:
        x = np.zeros(n, np.float32)
        x[j] = np.float32(3.0)
        want = (sc[:, j // 32] * q[:, j]).astype(np.float32) * np.float32(3.0)
        assert np.array_equal(gpu_matvec(q8d, w, x, n, p, canary=False), want), j


def test_matvec_mma_minus_128_and_sum_of_x(q8d):
    n, p = 2048, 2432
    w = synth.q8_const_matrix(p, n, 0x3C00, -128)
    assert np.array_equal(gpu_matvec(q8d, w, np.ones(n, np.float32), n, p),
                          np.full(p, -128.0 * n, np.float32))
    w1 = synth.q8_const_matrix(p, n, 0x3C00, 1)
    x = synth.normal_f32(13, "mms", n)
    got = gpu_matvec(q8d, w1, x, n, p)
    assert np.all(np.abs(got - np.sum(x, dtype=np.float64)) <= TOL * np.abs(x).sum())


def test_matvec_mma_wide_dynamic_range_and_determinism(q8d, orc):
    """x spanning 2^-20 .. 2^10 (the f16 split after the vector's power-of-two
    scale) within the bar; two launches agree bitwise."""
    n, p = 3584, 2600
    w = synth.q8_matrix(14, "mmr", p, n)
    x = synth.normal_f32(14, "mmrx", n) * np.exp2(synth.stream(14, "mmre").integers(-20, 11, n)).astype(np.float32)
    ref, ab = orc.q8_matvec(w, x, n, p)
    a = gpu_matvec(q8d, w, x, n, p)
    b = gpu_matvec(q8d, w, x, n, p)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.all(np.abs(a.astype(np.float64) - ref) <= TOL * ab), (np.abs(a - ref) / ab).max()


def test_matvec_mma_control_perturbed_byte(q8d):
    n, p = 2048, 2432
    w = synth.q8_matrix(15, "mmc", p, n)
    x = synth.normal_f32(15, "mmcx", n)
    a = gpu_matvec(q8d, w, x, n, p)
    w2 = w.copy()
    w2[1000, 34 * 37 + 9] ^= 0x11
    b = gpu_matvec(q8d, w2, x, n, p)
    assert a[1000] != b[1000] and np.array_equal(np.delete(a, 1000), np.delete(b, 1000))


# ---------------------------------------------------------------------------- launch chaining
def test_matvec_chain_without_sync(q8d, orc):
    """Calls on one stream, each reading the previous call's output, with no
    host synchronisation in between (the kernels are programmatic dependents
    of the one before): every call must see its input complete.  The
    intermediates start as NaN, so an early read would show."""
    n1, p1, p2, p3 = 3584, 3584, 896, 3584  # tensor-core, CUDA-core, CUDA-core kernels
    w1 = synth.q8_matrix(11, "chain.w1", p1, n1)
    w2 = synth.q8_matrix(11, "chain.w2", p2, p1)
    w3 = synth.q8_matrix(11, "chain.w3", p3, p2)
    x = synth.normal_f32(11, "chain.x", n1)
    xd, w1d, w2d, w3d = dev(x), dev(w1), dev(w2), dev(w3)
    y1 = torch.full((p1,), float("nan"), device="cuda")
    y2 = torch.full((p2,), float("nan"), device="cuda")
    y3 = torch.full((p3,), float("nan"), device="cuda")
    for _ in range(3):  # repeated: later chains overwrite live buffers
        q8d.q8d_matvec(xd, w1d, y1, n1, p1)
        q8d.q8d_matvec(y1, w2d, y2, p1, p2)
        q8d.q8d_matvec(y2, w3d, y3, p2, p3)
    torch.cuda.synchronize()
    g1, g2, g3 = y1.cpu().numpy(), y2.cpu().numpy(), y3.cpu().numpy()
    for w, xin, got, n, p in ((w1, x, g1, n1, p1), (w2, g1, g2, p1, p2), (w3, g2, g3, p2, p3)):
        ref, ab = orc.q8_matvec(w, xin, n, p)
        assert np.all(np.abs(got - ref) <= TOL * ab + 1e-30)


def test_small_m_chain_shared_workspace(q8d, orc):
    """Two tensor-core small-M calls back to back on one stream, sharing one
    workspace, the second reading the first's output as its activations:
    the second call's image kernel must wait until the first call's matmul
    no longer reads the workspace, and must see its output complete."""
    m, n1, p1, p2 = 16, 512, 512, 300
    w1 = synth.q8_matrix(12, "schain.w1", p1, n1)
    w2 = synth.q8_matrix(12, "schain.w2", p2, p1)
    X1 = synth.normal_f32(12, "schain.X", (m, n1))
    need = max(q8d.q8d_matmul_small_m_workspace_bytes(m, n1),
               q8d.q8d_matmul_small_m_workspace_bytes(m, p1))
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    Y1 = torch.full((m, p1), float("nan"), device="cuda")
    Y2 = torch.full((m, p2), float("nan"), device="cuda")
    w1d, w2d, X1d = dev(w1), dev(w2), dev(X1)
    for _ in range(3):
        q8d.q8d_matmul_small_m_ws(X1d, n1, w1d, Y1, p1, m, n1, p1, ws, need)
        q8d.q8d_matmul_small_m_ws(Y1, p1, w2d, Y2, p2, m, p1, p2, ws, need)
    torch.cuda.synchronize()
    G1, G2 = Y1.cpu().numpy(), Y2.cpu().numpy()
    ref1, ab1 = orc.q8_matmul(w1, X1, n1, p1)
    assert np.all(np.abs(G1 - ref1) <= TOL_TC * ab1)
    ref2, ab2 = orc.q8_matmul(w2, G1, p1, p2)
    assert np.all(np.abs(G2 - ref2) <= TOL_TC * ab2)
