"""q8d_kv_append and q8d_gqa_decode_attn (CUDA, through the C ABI) against
the oracle.  KV append and indexing: bit-exact.  Attention: per output
|gpu - oracle| <= 1e-5 * sum_t p_t |V_t|; L = 1 returns the V row bitwise."""
import math

import numpy as np
import pytest
import torch

import synth
from conftest import dev

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.mark.parametrize("dtype", [synth.KV_F16, synth.KV_F32])
@pytest.mark.parametrize("kvw,cap,pos", [(32, 8, 3), (1024, 16, 15), (512, 5, 0)])
def test_kv_append_bit_exact(q8d, orc, dtype, kvw, cap, pos):
    k = synth.normal_f32(1, "k", kvw) * 300   # exercises f16 overflow to inf and large values
    v = synth.normal_f32(1, "v", kvw) * 1e-5  # exercises f16 subnormals
    dt = np.float16 if dtype == synth.KV_F16 else np.float32
    kc0 = synth.normal_f32(2, "kc", (cap, kvw)).astype(dt)
    vc0 = synth.normal_f32(2, "vc", (cap, kvw)).astype(dt)
    kc_o, vc_o = kc0.copy(), vc0.copy()
    orc.kv_append(k, v, kc_o, vc_o, dtype, pos)
    kc, vc = dev(kc0), dev(vc0)
    d_pos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8d.q8d_kv_append(dev(k), dev(v), kc, vc, dtype, kvw, cap, d_pos, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    bits = np.uint16 if dtype == synth.KV_F16 else np.uint32
    assert np.array_equal(kc.cpu().numpy().view(bits), kc_o.view(bits))
    assert np.array_equal(vc.cpu().numpy().view(bits), vc_o.view(bits))


def test_kv_append_out_of_range_position_writes_nothing(q8d):
    kvw, cap = 64, 4
    kc = torch.ones((cap, kvw), dtype=torch.float16, device="cuda")
    vc = torch.ones((cap, kvw), dtype=torch.float16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (cap, -1, 1000):
        d_pos = torch.tensor([bad], dtype=torch.int32, device="cuda")
        q8d.q8d_kv_append(torch.zeros(kvw, device="cuda"), torch.zeros(kvw, device="cuda"), kc, vc,
                          q8d.Q8D_KV_F16, kvw, cap, d_pos, err)
    torch.cuda.synchronize()
    assert err.item() & q8d.Q8D_DERR_POS_RANGE
    assert torch.all(kc == 1) and torch.all(vc == 1)


def run_attn(q8d, q, kc, vc, dtype, H, Hk, D, lens, cap, scale, k_new=None, v_new=None,
             stride=None):
    batch = len(lens)
    kvw = Hk * D
    stride = cap * kvw if stride is None else stride
    ws_bytes = q8d.q8d_gqa_workspace_bytes(batch, H, Hk, D, cap)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((batch, H * D), -7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q8d.q8d_gqa_decode_attn(q, k_new, v_new, kc, vc, dtype, out, batch, H, Hk, D, cap, stride,
                            d_lens, scale, ws, ws_bytes, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), err.item()


CASES = [  # (H, Hk, D, dtype, L, cap)
    (16, 8, 128, synth.KV_F16, 512, 512),     # tiny config
    (4, 2, 16 * 4, synth.KV_F32, 9, 16),      # the pages' test shape at head_dim 64
    (14, 2, 64, synth.KV_F32, 512, 4096),     # Qwen2.5-0.5B-shaped
    (14, 2, 64, synth.KV_F32, 2048, 2048),
    (16, 8, 128, synth.KV_F16, 2048, 2048),   # Qwen3-0.6B-shaped
    (28, 4, 128, synth.KV_F16, 2048, 8192),   # 7B-shaped
    (28, 4, 128, synth.KV_F16, 8192, 8192),
    (6, 2, 64, synth.KV_F16, 129, 300),       # ragged: one row past a chunk
    (3, 3, 128, synth.KV_F32, 77, 77),
    (16, 1, 128, synth.KV_F16, 1000, 1000),   # group of 16
]


@pytest.mark.parametrize("H,Hk,D,dtype,L,cap", CASES)
def test_attention_parity(q8d, orc, H, Hk, D, dtype, L, cap):
    kvw = Hk * D
    q = synth.normal_f32(0, "attn.q", H * D)
    mk = synth.normal_f16 if dtype == synth.KV_F16 else synth.normal_f32
    kc = np.zeros((cap, kvw), mk(0, "z", 1).dtype)
    vc = np.zeros((cap, kvw), kc.dtype)
    kc[:L] = mk(0, "attn.k", (L, kvw))
    vc[:L] = mk(0, "attn.v", (L, kvw))
    scale = 1 / math.sqrt(D)
    ref, ab = orc.gqa_decode_attn(q, kc, vc, dtype, H, Hk, D, L, scale)
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), dtype, H, Hk, D, [L], cap, scale)
    assert err == 0
    assert np.all(np.abs(got[0] - ref) <= TOL * ab), (np.abs(got[0] - ref) / ab).max()


@pytest.mark.parametrize("dtype", [synth.KV_F16, synth.KV_F32])
def test_attention_single_position_is_v_row(q8d, dtype):
    H, Hk, D, cap = 28, 4, 128, 64
    mk = synth.normal_f16 if dtype == synth.KV_F16 else synth.normal_f32
    kc = mk(1, "k", (cap, Hk * D))
    vc = mk(1, "v", (cap, Hk * D))
    q = synth.normal_f32(1, "q", H * D) * 30
    got, _ = run_attn(q8d, dev(q), dev(kc), dev(vc), dtype, H, Hk, D, [1], cap, 0.1)
    for h in range(H):
        g = h // (H // Hk)
        assert np.array_equal(got[0, h * D:(h + 1) * D], vc[0, g * D:(g + 1) * D].astype(np.float32))


def test_attention_identical_keys_mean_v(q8d):
    H, Hk, D, L = 14, 2, 64, 3000
    krow = synth.normal_f32(2, "k", Hk * D)
    kc = np.tile(krow, (L, 1)).astype(np.float16)
    vc = synth.normal_f16(2, "v", (L, Hk * D))
    q = synth.normal_f32(2, "q", H * D)
    got, _ = run_attn(q8d, dev(q), dev(kc), dev(vc), synth.KV_F16, H, Hk, D, [L], L, 1 / 8)
    mean = vc.astype(np.float64).mean(axis=0)
    for h in range(H):
        g = h // (H // Hk)
        ab = np.abs(vc[:, g * D:(g + 1) * D].astype(np.float64)).mean(axis=0)
        assert np.all(np.abs(got[0, h * D:(h + 1) * D] - mean[g * D:(g + 1) * D]) <= TOL * ab)


def test_attention_in_kernel_append(q8d, orc):
    """k_new/v_new are written at row L-1 (rounded) and attended to; the
    cache afterwards equals q8d_kv_append's result bit for bit."""
    H, Hk, D, L, cap = 28, 4, 128, 700, 1024
    kvw = Hk * D
    kc = np.zeros((cap, kvw), np.float16)
    vc = np.zeros((cap, kvw), np.float16)
    kc[:L - 1] = synth.normal_f16(3, "k", (L - 1, kvw))
    vc[:L - 1] = synth.normal_f16(3, "v", (L - 1, kvw))
    kn = synth.normal_f32(3, "kn", kvw) * 3
    vn = synth.normal_f32(3, "vn", kvw) * 3
    q = synth.normal_f32(3, "q", H * D)
    kc_o, vc_o = kc.copy(), vc.copy()
    orc.kv_append(kn, vn, kc_o, vc_o, synth.KV_F16, L - 1)
    ref, ab = orc.gqa_decode_attn(q, kc_o, vc_o, synth.KV_F16, H, Hk, D, L, 1 / math.sqrt(D))
    kcd, vcd = dev(kc), dev(vc)
    got, err = run_attn(q8d, dev(q), kcd, vcd, synth.KV_F16, H, Hk, D, [L], cap, 1 / math.sqrt(D),
                        k_new=dev(kn), v_new=dev(vn))
    assert err == 0
    assert np.all(np.abs(got[0] - ref) <= TOL * ab)
    assert np.array_equal(kcd.cpu().numpy().view(np.uint16), kc_o.view(np.uint16))
    assert np.array_equal(vcd.cpu().numpy().view(np.uint16), vc_o.view(np.uint16))


def test_attention_split_invariance(q8d):
    """The chunk count follows cap; results for different chunkings agree
    within the tolerance (the split is invisible up to rounding)."""
    H, Hk, D, L = 28, 4, 128, 5000
    kvw = Hk * D
    outs = []
    for cap in (5000, 16384, 65536):
        kc = np.zeros((cap, kvw), np.float16)
        vc = np.zeros((cap, kvw), np.float16)
        kc[:L] = synth.normal_f16(4, "k", (L, kvw))
        vc[:L] = synth.normal_f16(4, "v", (L, kvw))
        got, _ = run_attn(q8d, dev(synth.normal_f32(4, "q", H * D)), dev(kc), dev(vc),
                          synth.KV_F16, H, Hk, D, [L], cap, 0.0884)
        outs.append(got[0])
    ab = np.abs(synth.normal_f16(4, "v", (L, kvw))).astype(np.float64).max()
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2 * TOL * ab


def test_attention_ragged_batch_32768(q8d, orc):
    """Stress: 8 sequences of 7B heads, lengths uniform in [1, 32768], one
    cache of 32768 rows per sequence; every output checked."""
    H, Hk, D, cap = 28, 4, 128, 32768
    kvw = Hk * D
    lens = synth.stream(0, "ragged.lens").integers(1, cap + 1, 8).tolist()
    lens[0] = 1
    kc = np.zeros((8, cap, kvw), np.float16)
    vc = np.zeros((8, cap, kvw), np.float16)
    for s, L in enumerate(lens):
        kc[s, :L] = synth.normal_f16(s, "ragged.k", (L, kvw))
        vc[s, :L] = synth.normal_f16(s, "ragged.v", (L, kvw))
    q = synth.normal_f32(0, "ragged.q", (8, H * D))
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), synth.KV_F16, H, Hk, D, lens, cap,
                        1 / math.sqrt(D))
    assert err == 0
    for s, L in enumerate(lens):
        ref, ab = orc.gqa_decode_attn(q[s], kc[s], vc[s], synth.KV_F16, H, Hk, D, L, 1 / math.sqrt(D))
        assert np.all(np.abs(got[s] - ref) <= TOL * ab), (s, L)


@pytest.mark.parametrize("dtype", [synth.KV_F16, synth.KV_F32])
def test_attention_one_long_sequence_among_short_ones(q8d, orc, dtype):
    """Length-proportional split at its clamp: one 32768-row sequence next to
    seven 1-row ones wants ~144 chunks and gets the workspace's slots."""
    H, Hk, D, cap = 28, 4, 128, 32768
    kvw = Hk * D
    lens = [cap, 1, 1, 1, 1, 1, 1, 1]
    npdt = np.float16 if dtype == synth.KV_F16 else np.float32
    kc = np.zeros((8, cap, kvw), npdt)
    vc = np.zeros((8, cap, kvw), npdt)
    for s_, L in enumerate(lens):
        kc[s_, :L] = synth.normal_f16(s_, "long.k", (L, kvw)).astype(npdt)
        vc[s_, :L] = synth.normal_f16(s_, "long.v", (L, kvw)).astype(npdt)
    q = synth.normal_f32(0, "long.q", (8, H * D))
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), dtype, H, Hk, D, lens, cap,
                        1 / math.sqrt(D))
    assert err == 0
    for s_, L in enumerate(lens):
        ref, ab = orc.gqa_decode_attn(q[s_], kc[s_], vc[s_], dtype, H, Hk, D, L, 1 / math.sqrt(D))
        assert np.all(np.abs(got[s_] - ref) <= TOL * ab), (s_, L)


def test_attention_batch_larger_than_the_chunk_grid(q8d, orc):
    """160 sequences (more than the chunk CTAs a KV head would get): one CTA
    per sequence; lengths 1..160 (seeded order), every output checked."""
    H, Hk, D, cap = 8, 4, 64, 200
    kvw = Hk * D
    batch = 160
    lens = (synth.stream(0, "wide.lens").permutation(batch) + 1).tolist()
    kc = synth.normal_f16(0, "wide.k", (batch, cap, kvw))
    vc = synth.normal_f16(0, "wide.v", (batch, cap, kvw))
    q = synth.normal_f32(0, "wide.q", (batch, H * D))
    got, err = run_attn(q8d, dev(q), dev(kc), dev(vc), synth.KV_F16, H, Hk, D, lens, cap, 0.125)
    assert err == 0
    for s_, L in enumerate(lens):
        ref, ab = orc.gqa_decode_attn(q[s_], kc[s_], vc[s_], synth.KV_F16, H, Hk, D, L, 0.125)
        assert np.all(np.abs(got[s_] - ref) <= TOL * ab), (s_, L)


def test_attention_bad_length_sets_error_and_nan(q8d):
    H, Hk, D, cap = 4, 2, 64, 32
    kc = torch.zeros((2, cap, Hk * D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.zeros((2, H * D), device="cuda")
    got, err = run_attn(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [5, cap + 1], cap, 0.125)
    assert err & q8d.Q8D_DERR_LEN_RANGE
    assert np.isnan(got[1]).all() and np.isfinite(got[0]).all()
    got, err = run_attn(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [0, 3], cap, 0.125)
    assert err & q8d.Q8D_DERR_LEN_RANGE and np.isnan(got[0]).all()


def test_attention_control_shifted_length_changes_output(q8d):
    H, Hk, D, cap = 16, 8, 128, 600
    kc = dev(synth.normal_f16(5, "k", (cap, Hk * D)))
    vc = dev(synth.normal_f16(5, "v", (cap, Hk * D)))
    q = dev(synth.normal_f32(5, "q", H * D))
    a, _ = run_attn(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [500], cap, 0.088)
    b, _ = run_attn(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [501], cap, 0.088)
    c, _ = run_attn(q8d, q, kc, vc, synth.KV_F16, H, Hk, D, [500], cap, 0.088)
    assert not np.array_equal(a, b)
    assert np.array_equal(a.view(np.uint32), c.view(np.uint32))  # deterministic


# ---------------------------------------------------------------------------- launch chaining
@pytest.mark.parametrize("dtype,noalloc", [(synth.KV_F16, False), (synth.KV_F32, False),
                                           (synth.KV_Q8_0, False), (synth.KV_F16, True)])
def test_attention_chain_without_sync(q8d, orc, dtype, noalloc):
    """Three decode-like rounds on one stream with no host synchronisation:
    matvecs make q, k and v from x, attention appends k and v at row L-1 and
    attends, and its output is the next round's x.  The attention kernels
    and their combine are programmatic dependents of the kernels before
    them, and every round reuses one workspace: each call must see its
    inputs (activations, the rows appended by the previous round) complete
    and must not overwrite partials the previous combine still reads.
    Intermediates start as NaN, so an early read would show."""
    H, Hk, D, L0, cap = 28, 4, 128, 300, 512
    n, kvw, rounds = H * D, Hk * D, 3
    # block scales ~1/(E|q| sqrt(n)): q, k, v keep x's magnitude round after
    # round (no growth into f16 overflow)
    wq = synth.q8_matrix(21, "achain.wq", n, n, 1e-4, 3e-4)
    wk = synth.q8_matrix(21, "achain.wk", kvw, n, 1e-4, 3e-4)
    wv = synth.q8_matrix(21, "achain.wv", kvw, n, 1e-4, 3e-4)
    x0 = synth.normal_f32(21, "achain.x", n)
    if dtype == synth.KV_Q8_0:  # packed rows of 34-byte blocks
        kc = synth.q8_kv_cache(21, "achain.kq", cap, kvw)
        vc = synth.q8_kv_cache(21, "achain.vq", cap, kvw)
    else:
        npdt = np.float16 if dtype == synth.KV_F16 else np.float32
        kc = np.zeros((cap, kvw), npdt)
        vc = np.zeros((cap, kvw), npdt)
        kc[:L0 - 1] = synth.normal_f16(21, "achain.k", (L0 - 1, kvw))
        vc[:L0 - 1] = synth.normal_f16(21, "achain.v", (L0 - 1, kvw))
    kc0, vc0 = kc.copy(), vc.copy()
    wqd, wkd, wvd, kcd, vcd = dev(wq), dev(wk), dev(wv), dev(kc), dev(vc)
    nan = lambda m: torch.full((m,), float("nan"), device="cuda")
    xs = [dev(x0)] + [nan(n) for _ in range(rounds)]  # xs[r + 1]: round r's attention output
    qs, ks, vs = [nan(n) for _ in range(rounds)], [nan(kvw) for _ in range(rounds)], \
        [nan(kvw) for _ in range(rounds)]
    lens = [torch.tensor([L0 + r], dtype=torch.int32, device="cuda") for r in range(rounds)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(D)
    ws_bytes = q8d.q8d_gqa_workspace_bytes(1, H, Hk, D, cap)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for r in range(rounds):
        q8d.q8d_matvec(xs[r], wqd, qs[r], n, n)
        q8d.q8d_matvec(xs[r], wkd, ks[r], n, kvw)
        q8d.q8d_matvec(xs[r], wvd, vs[r], n, kvw)
        args = (qs[r], ks[r], vs[r], kcd, vcd, dtype, xs[r + 1], 1, H, Hk, D, cap, cap * kvw, lens[r],
                scale)
        if noalloc:
            q8d.q8d_gqa_decode_attn_noalloc(*args, err)
        else:
            q8d.q8d_gqa_decode_attn(*args, ws, ws_bytes, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = [t.cpu().numpy() for t in xs]
    kc_o, vc_o = kc0.copy(), vc0.copy()
    for r in range(rounds):
        q_g, k_g, v_g = qs[r].cpu().numpy(), ks[r].cpu().numpy(), vs[r].cpu().numpy()
        for w, g, p in ((wq, q_g, n), (wk, k_g, kvw), (wv, v_g, kvw)):
            ref, ab = orc.q8_matvec(w, got[r], n, p)
            assert np.all(np.abs(g - ref) <= TOL * ab + 1e-30)
        orc.kv_append(k_g, v_g, kc_o, vc_o, dtype, L0 - 1 + r)
        ref, ab = orc.gqa_decode_attn(q_g, kc_o, vc_o, dtype, H, Hk, D, L0 + r, scale)
        assert np.all(np.abs(got[r + 1] - ref) <= TOL * ab)
    bits = {synth.KV_F16: np.uint16, synth.KV_F32: np.uint32, synth.KV_Q8_0: np.uint8}[dtype]
    assert np.array_equal(kcd.cpu().numpy().view(bits), kc_o.view(bits))
    assert np.array_equal(vcd.cpu().numpy().view(bits), vc_o.view(bits))
