"""Packed Q8_0 KV cache (Q8D_KV_Q8_0) through the C ABI against the oracle
("minfer Metal Backend Design", "Execution dispatch": packed q8_0 KV; the
store is byte-identical to the CPU quantizer, decode reads the blocks
natively).  Store: bit-exact bytes.  Attention: per output
|gpu - oracle| <= 1e-5 * sum_t p_t |V_t| on the same packed bytes; L = 1
returns the dequantised V row bitwise."""
import math

import numpy as np
import pytest
import torch

import synth
from conftest import dev

pytestmark = pytest.mark.gpu
TOL = 1e-5
Q8 = synth.KV_Q8_0


def rb(kvw):
    return kvw // 32 * 34


def append_inputs(kvw, seed):
    """k, v rows mixing magnitudes, an all-zero block, and blocks whose
    quantisation hits exact halves (amax 127 makes d = 1)."""
    k = synth.normal_f32(seed, "q8a.k", kvw) * np.float32(300.0)
    v = synth.normal_f32(seed, "q8a.v", kvw) * np.float32(1e-5)
    if kvw >= 96:
        k[32:64] = 0.0
        halves = np.array([127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5] * 4, np.float32)
        v[64:96] = halves
    return k, v


@pytest.mark.parametrize("kvw,cap,pos", [(32, 8, 3), (128, 16, 15), (512, 5, 0), (1024, 9, 7)])
def test_q8kv_append_bit_exact(q8d, orc, kvw, cap, pos):
    k, v = append_inputs(kvw, 1)
    kc0 = synth.q8_kv_cache(2, "q8a.kc", cap, kvw)
    vc0 = synth.q8_kv_cache(2, "q8a.vc", cap, kvw)
    kc_o, vc_o = kc0.copy(), vc0.copy()
    orc.kv_append(k, v, kc_o, vc_o, Q8, pos)
    kc, vc = dev(kc0), dev(vc0)
    d_pos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8d.q8d_kv_append(dev(k), dev(v), kc, vc, Q8, kvw, cap, d_pos, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(kc.cpu().numpy(), kc_o)
    assert np.array_equal(vc.cpu().numpy(), vc_o)


def test_q8kv_append_random_rows_bit_exact(q8d, orc):
    """Many rows of N(0, sigma) values at several scales, one call per row."""
    kvw, cap = 512, 24
    kc = torch.zeros((cap, rb(kvw)), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    kc_o = np.zeros((cap, rb(kvw)), np.uint8)
    vc_o = np.zeros_like(kc_o)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for pos in range(cap):
        sig = np.float32(10.0 ** (pos % 8 - 4))
        k = synth.normal_f32(pos, "q8r.k", kvw) * sig
        v = synth.normal_f32(pos, "q8r.v", kvw) * sig
        orc.kv_append(k, v, kc_o, vc_o, Q8, pos)
        d_pos = torch.tensor([pos], dtype=torch.int32, device="cuda")
        q8d.q8d_kv_append(dev(k), dev(v), kc, vc, Q8, kvw, cap, d_pos, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(kc.cpu().numpy(), kc_o) and np.array_equal(vc.cpu().numpy(), vc_o)


def test_q8kv_append_out_of_range_position_writes_nothing(q8d):
    kvw, cap = 64, 4
    kc = torch.full((cap, rb(kvw)), 5, dtype=torch.uint8, device="cuda")
    vc = torch.full((cap, rb(kvw)), 5, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (cap, -1):
        d_pos = torch.tensor([bad], dtype=torch.int32, device="cuda")
        q8d.q8d_kv_append(torch.ones(kvw, device="cuda"), torch.ones(kvw, device="cuda"), kc, vc,
                          Q8, kvw, cap, d_pos, err)
    torch.cuda.synchronize()
    assert err.item() & q8d.Q8D_DERR_POS_RANGE
    assert torch.all(kc == 5) and torch.all(vc == 5)


def run_attn(q8d, q, kc, vc, H, Hk, D, lens, cap, scale, k_new=None, v_new=None):
    batch = len(lens)
    ws_bytes = q8d.q8d_gqa_workspace_bytes(batch, H, Hk, D, cap)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((batch, H * D), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q8d.q8d_gqa_decode_attn(q, k_new, v_new, kc, vc, Q8, out, batch, H, Hk, D, cap, cap * Hk * D,
                            d_lens, scale, ws, ws_bytes, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), err.item()


CASES = [  # (H, Hk, D, L, cap)
    (16, 8, 128, 512, 512),
    (4, 2, 64, 9, 16),
    (14, 2, 64, 2048, 2048),
    (16, 8, 128, 2048, 2048),
    (28, 4, 128, 2048, 8192),
    (28, 4, 128, 8192, 8192),
    (6, 2, 64, 129, 300),
    (16, 1, 128, 1000, 1000),
    (3, 3, 128, 77, 80),
]


@pytest.mark.parametrize("H,Hk,D,L,cap", CASES)
def test_q8kv_attention_parity(q8d, orc, H, Hk, D, L, cap):
    kvw = Hk * D
    q = synth.normal_f32(0, "q8.q", H * D)
    kc = synth.q8_kv_cache(0, "q8.k", cap, kvw, L)
    vc = synth.q8_kv_cache(0, "q8.v", cap, kvw, L)
    scale = 1 / math.sqrt(D)
    ref, ab = orc.gqa_decode_attn(q, kc, vc, Q8, H, Hk, D, L, scale)
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), H, Hk, D, [L], cap, scale)
    assert err == 0
    assert np.all(np.abs(got[0] - ref) <= TOL * ab), (np.abs(got[0] - ref) / ab).max()


def dequant(c, rows, kvw):
    blk = c[:rows].reshape(rows, kvw // 32, 34)
    sc = blk[:, :, 0:2].copy().view("<f2")[..., 0].astype(np.float32)
    q = blk[:, :, 2:].view(np.int8).astype(np.float32)
    return (sc[:, :, None] * q).reshape(rows, kvw)


@pytest.mark.parametrize("D", [64, 128])
def test_q8kv_single_position_is_dequantized_v_row(q8d, D):
    H, Hk, cap = 28, 4, 64
    kc = synth.q8_kv_cache(1, "q8.k1", cap, Hk * D)
    vc = synth.q8_kv_cache(1, "q8.v1", cap, Hk * D)
    q = synth.normal_f32(1, "q8.q1", H * D) * 30
    got, _ = run_attn(q8d, dev(q), dev(kc), dev(vc), H, Hk, D, [1], cap, 0.1)
    v0 = dequant(vc, 1, Hk * D)[0]
    for h in range(H):
        g = h // (H // Hk)
        assert np.array_equal(got[0, h * D:(h + 1) * D], v0[g * D:(g + 1) * D])


@pytest.mark.parametrize("lo,hi", [(1e-7, 5e-7), (50.0, 4000.0), (1e-3, 2e3)])
def test_q8kv_attention_extreme_v_scales(q8d, orc, lo, hi):
    """V block scales far from the usual range, and spread over six decades
    in one cache: the per-warp range factor keeps P * scale inside f16."""
    H, Hk, D, L = 14, 2, 128, 700
    kvw = Hk * D
    q = synth.normal_f32(3, "q8x.q", H * D)
    kc = synth.q8_kv_cache(3, "q8x.k", L, kvw)
    vc = synth.q8_matrix(3, f"q8x.v{lo}", L, kvw, lo, hi)
    ref, ab = orc.gqa_decode_attn(q, kc, vc, Q8, H, Hk, D, L, 1 / math.sqrt(D))
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), H, Hk, D, [L], L, 1 / math.sqrt(D))
    assert err == 0
    assert np.all(np.abs(got[0] - ref) <= TOL * ab), (np.abs(got[0] - ref) / ab).max()


def test_q8kv_attention_zero_values(q8d):
    H, Hk, D, L = 8, 2, 64, 300
    kc = synth.q8_kv_cache(4, "q8z.k", L, Hk * D)
    vc = np.zeros((L, rb(Hk * D)), np.uint8)
    got, err = run_attn(q8d, dev(synth.normal_f32(4, "q8z.q", H * D)), dev(kc), dev(vc), H, Hk, D,
                        [L], L, 0.125)
    assert err == 0 and np.array_equal(got, np.zeros_like(got))


def test_q8kv_in_kernel_append(q8d, orc):
    """k_new/v_new are quantized into row L-1 by the store quantizer and
    attended to; the cache afterwards equals the oracle's append bytes."""
    H, Hk, D, L, cap = 28, 4, 128, 700, 1024
    kvw = Hk * D
    kc = synth.q8_kv_cache(5, "q8i.k", cap, kvw, L - 1)
    vc = synth.q8_kv_cache(5, "q8i.v", cap, kvw, L - 1)
    kn = synth.normal_f32(5, "q8i.kn", kvw) * 3
    vn = synth.normal_f32(5, "q8i.vn", kvw) * 3
    q = synth.normal_f32(5, "q8i.q", H * D)
    kc_o, vc_o = kc.copy(), vc.copy()
    orc.kv_append(kn, vn, kc_o, vc_o, Q8, L - 1)
    ref, ab = orc.gqa_decode_attn(q, kc_o, vc_o, Q8, H, Hk, D, L, 1 / math.sqrt(D))
    kcd, vcd = dev(kc), dev(vc)
    got, err = run_attn(q8d, dev(q), kcd, vcd, H, Hk, D, [L], cap, 1 / math.sqrt(D),
                        k_new=dev(kn), v_new=dev(vn))
    assert err == 0
    assert np.all(np.abs(got[0] - ref) <= TOL * ab)
    assert np.array_equal(kcd.cpu().numpy(), kc_o) and np.array_equal(vcd.cpu().numpy(), vc_o)


def test_q8kv_ragged_batch(q8d, orc):
    """8 sequences of 7B heads with seeded ragged lengths up to 8192 (one
    of length 1), one packed cache of 8192 rows per sequence."""
    H, Hk, D, cap = 28, 4, 128, 8192
    kvw = Hk * D
    lens = synth.stream(0, "ragged.lens.q8").integers(1, cap + 1, 8).tolist()
    lens[0] = 1
    kc = np.stack([synth.q8_kv_cache(s, "q8b.k", cap, kvw, L) for s, L in enumerate(lens)])
    vc = np.stack([synth.q8_kv_cache(s, "q8b.v", cap, kvw, L) for s, L in enumerate(lens)])
    q = synth.normal_f32(0, "q8b.q", (8, H * D))
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), H, Hk, D, lens, cap, 1 / math.sqrt(D))
    assert err == 0
    for s, L in enumerate(lens):
        ref, ab = orc.gqa_decode_attn(q[s], kc[s], vc[s], Q8, H, Hk, D, L, 1 / math.sqrt(D))
        assert np.all(np.abs(got[s] - ref) <= TOL * ab), (s, L)


def test_q8kv_split_invariance(q8d):
    H, Hk, D, L = 28, 4, 128, 5000
    kvw = Hk * D
    q = synth.normal_f32(6, "q8s.q", H * D)
    outs = []
    for cap in (5000, 16384, 65536):
        kc = synth.q8_kv_cache(6, "q8s.k", cap, kvw, L)
        vc = synth.q8_kv_cache(6, "q8s.v", cap, kvw, L)
        got, _ = run_attn(q8d, dev(q), dev(kc), dev(vc), H, Hk, D, [L], cap, 0.0884)
        outs.append(got[0])
    vmax = np.abs(dequant(synth.q8_kv_cache(6, "q8s.v", L, kvw), L, kvw)).max()
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2 * TOL * vmax


def test_q8kv_bad_length_sets_error_and_nan(q8d):
    H, Hk, D, cap = 8, 2, 64, 64
    kc = synth.q8_kv_cache(7, "q8e.k", cap, Hk * D)
    vc = synth.q8_kv_cache(7, "q8e.v", cap, Hk * D)
    got, err = run_attn(q8d, dev(synth.normal_f32(7, "q8e.q", H * D)), dev(kc), dev(vc), H, Hk, D,
                        [cap + 1], cap, 0.125)
    assert err & q8d.Q8D_DERR_LEN_RANGE and np.isnan(got).all()


def test_q8kv_control_changed_block_changes_output(q8d):
    """A changed quant byte of one cached V row must change the output of its
    KV head's query heads only (guards a vacuous gate)."""
    H, Hk, D, L = 8, 2, 64, 200
    kvw = Hk * D
    q = synth.normal_f32(8, "q8c.q", H * D)
    kc = synth.q8_kv_cache(8, "q8c.k", L, kvw)
    vc = synth.q8_kv_cache(8, "q8c.v", L, kvw)
    a, _ = run_attn(q8d, dev(q), dev(kc), dev(vc), H, Hk, D, [L], L, 0.125)
    vc2 = vc.copy()
    vc2[77, 2 * 34 + 5] ^= 0x21  # KV head 1 (blocks 2, 3), quant 3 of block 2
    b, _ = run_attn(q8d, dev(q), dev(kc), dev(vc2), H, Hk, D, [L], L, 0.125)
    G = H // Hk
    assert np.array_equal(a[0, :G * D], b[0, :G * D])
    assert not np.array_equal(a[0, G * D:], b[0, G * D:])
