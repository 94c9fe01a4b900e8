"""q8d_gqa_decode_attn_window (CUDA, through the C ABI) against the oracle's
windowed attention ("minfer Metal Backend Design", "Execution dispatch",
window modes: explicit [lo, hi) spans and (cell, len) run maps).  Gates as
the pages name them: a one-cell window returns that cell's V row bitwise, a
window shifted by one cell and a wrong shared base change the output; every
other window within 1e-5 * sum_t p_t |V_t| per output."""
import math

import numpy as np
import pytest
import torch

import synth
from conftest import dev

pytestmark = pytest.mark.gpu
TOL = 1e-5
DTYPES = [synth.KV_F16, synth.KV_F32, synth.KV_Q8_0]


def make_cache(dtype, seed, name, cap, kvw):
    if dtype == synth.KV_Q8_0:
        return synth.q8_kv_cache(seed, name, cap, kvw)
    if dtype == synth.KV_F16:
        return synth.normal_f16(seed, name, (cap, kvw))
    return synth.normal_f32(seed, name, (cap, kvw))


def runs_array(runs_per_seq):
    a = np.zeros((len(runs_per_seq), 4, 2), np.int32)
    for s, runs in enumerate(runs_per_seq):
        for r, (cell, ln) in enumerate(runs):
            a[s, r] = (cell, ln)
    return a


def run_window(q8d, q, kc, vc, dtype, H, Hk, D, runs_per_seq, cap, stride, scale, k_new=None,
               v_new=None):
    batch = len(runs_per_seq)
    ws_bytes = q8d.q8d_gqa_workspace_bytes(batch, H, Hk, D, cap)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((batch, H * D), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_runs = dev(runs_array(runs_per_seq))
    q8d.q8d_gqa_decode_attn_window(q, k_new, v_new, kc, vc, dtype, out, batch, H, Hk, D, cap,
                                   stride, d_runs, scale, ws, ws_bytes, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), err.item()


def v_row(vc, dtype, cell, kvw):
    if dtype == synth.KV_Q8_0:
        blk = vc[cell].reshape(kvw // 32, 34)
        sc = blk[:, 0:2].copy().view("<f2")[:, 0].astype(np.float32)
        return (sc[:, None] * blk[:, 2:].view(np.int8).astype(np.float32)).ravel()
    return vc[cell].astype(np.float32)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,Hk,D", [(28, 4, 128), (6, 2, 64)])
def test_window_one_cell_is_that_v_row(q8d, dtype, H, Hk, D):
    cap = 300
    kvw = Hk * D
    kc = make_cache(dtype, 1, "w1.k", cap, kvw)
    vc = make_cache(dtype, 1, "w1.v", cap, kvw)
    q = synth.normal_f32(1, "w1.q", (3, H * D)) * 30
    cells = [0, 157, cap - 1]
    got, err = run_window(q8d, dev(q), dev(kc), dev(vc), dtype, H, Hk, D,
                          [[(c, 1)] for c in cells], cap, 0, 0.1)
    assert err == 0
    for s, c in enumerate(cells):
        v = v_row(vc, dtype, c, kvw)
        for h in range(H):
            g = h // (H // Hk)
            assert np.array_equal(got[s, h * D:(h + 1) * D], v[g * D:(g + 1) * D]), (s, c, h)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("lo,hi", [(0, 700), (1000, 5000), (333, 334 + 64), (4095, 6000)])
def test_window_span_parity(q8d, orc, dtype, lo, hi):
    H, Hk, D, cap = 28, 4, 128, 6000
    kvw = Hk * D
    kc = make_cache(dtype, 2, "ws.k", cap, kvw)
    vc = make_cache(dtype, 2, "ws.v", cap, kvw)
    q = synth.normal_f32(2, "ws.q", H * D)
    ref, ab = orc.gqa_decode_attn_runs(q, kc, vc, dtype, H, Hk, D, [(lo, hi - lo)], 1 / math.sqrt(D))
    got, err = run_window(q8d, dev(q), dev(kc), dev(vc), dtype, H, Hk, D, [[(lo, hi - lo)]], cap, 0,
                          1 / math.sqrt(D))
    assert err == 0
    assert np.all(np.abs(got[0] - ref) <= TOL * ab), (np.abs(got[0] - ref) / ab).max()


@pytest.mark.parametrize("dtype", DTYPES)
def test_window_shared_prefix_batch(q8d, orc, dtype):
    """Four sequences read one cache (stride 0): a shared prefix run plus a
    private run each, adjacent for one and gapped for the others."""
    H, Hk, D, cap = 14, 2, 64, 4096
    kvw = Hk * D
    kc = make_cache(dtype, 3, "wp.k", cap, kvw)
    vc = make_cache(dtype, 3, "wp.v", cap, kvw)
    q = synth.normal_f32(3, "wp.q", (4, H * D))
    pre = 1500
    maps = [[(0, pre), (pre, 300)], [(0, pre), (2000, 17)], [(0, pre), (2100, 1990)],
            [(0, pre), (3000, 1), (3500, 200), (4000, 96)]]
    got, err = run_window(q8d, dev(q), dev(kc), dev(vc), dtype, H, Hk, D, maps, cap, 0,
                          1 / math.sqrt(D))
    assert err == 0
    for s, m in enumerate(maps):
        ref, ab = orc.gqa_decode_attn_runs(q[s], kc, vc, dtype, H, Hk, D, m, 1 / math.sqrt(D))
        assert np.all(np.abs(got[s] - ref) <= TOL * ab), s


@pytest.mark.parametrize("dtype", [synth.KV_F16, synth.KV_Q8_0])
def test_window_full_span_equals_causal_call(q8d, dtype):
    """The span [0, L) takes the causal call's split and matches it bitwise."""
    H, Hk, D, L, cap = 28, 4, 128, 3000, 4096
    kvw = Hk * D
    kc = dev(make_cache(dtype, 4, "wc.k", cap, kvw))
    vc = dev(make_cache(dtype, 4, "wc.v", cap, kvw))
    q = dev(synth.normal_f32(4, "wc.q", H * D))
    got, _ = run_window(q8d, q, kc, vc, dtype, H, Hk, D, [[(0, L)]], cap, 0, 0.0884)
    ws_bytes = q8d.q8d_gqa_workspace_bytes(1, H, Hk, D, cap)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.empty((1, H * D), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8d.q8d_gqa_decode_attn(q, None, None, kc, vc, dtype, out, 1, H, Hk, D, cap, 0,
                            torch.tensor([L], dtype=torch.int32, device="cuda"), 0.0884, ws,
                            ws_bytes, err)
    torch.cuda.synchronize()
    assert np.array_equal(got, out.cpu().numpy())


def test_window_controls_shift_and_wrong_base_change_the_output(q8d):
    H, Hk, D, cap = 8, 2, 64, 500
    kvw = Hk * D
    kc = dev(make_cache(synth.KV_F16, 5, "wx.k", cap, kvw))
    vc = dev(make_cache(synth.KV_F16, 5, "wx.v", cap, kvw))
    q = dev(synth.normal_f32(5, "wx.q", H * D))
    base, _ = run_window(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [[(0, 100), (200, 50)]], cap, 0, 0.1)
    shifted, _ = run_window(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [[(0, 100), (201, 50)]], cap, 0, 0.1)
    wrong_base, _ = run_window(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [[(1, 100), (200, 50)]], cap, 0,
                               0.1)
    assert not np.array_equal(base, shifted)
    assert not np.array_equal(base, wrong_base)


@pytest.mark.parametrize("dtype", DTYPES)
def test_window_append_writes_the_last_window_row(q8d, orc, dtype):
    """k_new/v_new land on the last row of each sequence's window (its last
    non-empty run) exactly as q8d_kv_append would write them, and are
    attended to; per-sequence caches."""
    H, Hk, D, cap = 28, 4, 128, 1024
    kvw = Hk * D
    maps = [[(0, 300), (600, 41)], [(10, 1)], [(5, 500), (700, 0), (900, 3)]]
    B = len(maps)
    kc = np.stack([make_cache(dtype, 6 + s, "wa.k", cap, kvw) for s in range(B)])
    vc = np.stack([make_cache(dtype, 6 + s, "wa.v", cap, kvw) for s in range(B)])
    kn = synth.normal_f32(6, "wa.kn", (B, kvw)) * 2
    vn = synth.normal_f32(6, "wa.vn", (B, kvw)) * 2
    q = synth.normal_f32(6, "wa.q", (B, H * D))
    kcd, vcd = dev(kc), dev(vc)
    got, err = run_window(q8d, dev(q), kcd, vcd, dtype, H, Hk, D, maps, cap, cap * kvw,
                          1 / math.sqrt(D), k_new=dev(kn), v_new=dev(vn))
    assert err == 0
    kc_after, vc_after = kcd.cpu().numpy(), vcd.cpu().numpy()
    for s, m in enumerate(maps):
        last = [(c, n) for c, n in m if n > 0][-1]
        row = last[0] + last[1] - 1
        ko, vo = kc[s].copy(), vc[s].copy()
        orc.kv_append(kn[s], vn[s], ko, vo, dtype, row)
        assert np.array_equal(kc_after[s].view(np.uint8), ko.view(np.uint8)), s
        assert np.array_equal(vc_after[s].view(np.uint8), vo.view(np.uint8)), s
        ref, ab = orc.gqa_decode_attn_runs(q[s], ko, vo, dtype, H, Hk, D, m, 1 / math.sqrt(D))
        assert np.all(np.abs(got[s] - ref) <= TOL * ab), s


def test_window_bad_runs_flag_error_and_nan_only_there(q8d, orc):
    H, Hk, D, cap = 8, 2, 64, 200
    kvw = Hk * D
    kc = make_cache(synth.KV_F16, 7, "wb.k", cap, kvw)
    vc = make_cache(synth.KV_F16, 7, "wb.v", cap, kvw)
    q = synth.normal_f32(7, "wb.q", (4, H * D))
    maps = [[(0, 50)], [(190, 11)], [(0, 0)], [(-1, 5)]]
    got, err = run_window(q8d, dev(q), dev(kc), dev(vc), synth.KV_F16, H, Hk, D, maps, cap, 0, 0.125)
    assert err & q8d.Q8D_DERR_LEN_RANGE
    ref, ab = orc.gqa_decode_attn_runs(q[0], kc, vc, synth.KV_F16, H, Hk, D, maps[0], 0.125)
    assert np.all(np.abs(got[0] - ref) <= TOL * ab)
    assert np.isnan(got[1:]).all()
