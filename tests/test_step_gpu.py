"""The captured decode step (q8d_step_*) against the oracle's double-precision
step ("IV.4: One command buffer per token", "One command buffer": the
decode step attends seq = pos + 1 rows).  Named tolerance class for a whole
step (28 layers of f32 against f64): |logit_gpu - logit_oracle| <= 1e-3 *
max|logit_oracle|; the argmax must agree unless the oracle's top-2 gap is
inside that bound.  Appended KV rows: layer 0's at the kernel bar (the
matvec's 1e-5 * sum|terms| carried through bias, QK-norm and RoPE, plus one
f16 rounding for an f16 cache); later layers' within one f16 rounding plus
the step class relative to the row's RMS (their inputs carry the residual
stream's rounding, as the logits do)."""
import functools

import numpy as np
import pytest
import torch

import synth
from q8_block_quantized_matvec_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu
STEP_TOL = 1e-3
U32 = 2.0 ** -24  # f32 unit roundoff


def compare_step(logits_gpu, logits_ref, tok_gpu, tok_ref):
    scale = np.max(np.abs(logits_ref))
    err = np.max(np.abs(logits_gpu.astype(np.float64) - logits_ref))
    assert err <= STEP_TOL * scale, (err, scale)
    if tok_gpu != tok_ref:
        top = np.sort(logits_ref.astype(np.float64))[-2:]
        assert top[1] - top[0] <= 2 * STEP_TOL * scale, "argmax differs on a clear winner"
    return err / scale


def layer0_kv_bound(orc, w, shape, token, pos):
    """Layer 0's appended K and V rows recomputed in double from the oracle's
    parts (embedding row, RMSNorm), with a per-element bound on the f32
    step's deviation before the cache rounding: the matvec bar (1e-5 *
    sum|terms| per output) carried through the bias add, the per-head
    RMSNorm (first order) and the RoPE rotation, plus four f32 roundings of
    each step's result.  Layer 0 reads only the embedding row, so nothing
    upstream carries the step's accumulated rounding.
    Returns (k, k_err, v, v_err), float64 [kv_width]."""
    s = shape
    L0 = w.layers[0]
    xn = orc.rmsnorm(orc.dequant_row(w.embed, token, s.hidden), L0["attn_norm"], s.rms_eps)

    def proj(wq8, bias):
        W = np.stack([orc.dequant_row(wq8, r, s.hidden) for r in range(s.kv_width)])
        val = W @ xn
        err = 1e-5 * (np.abs(W) @ np.abs(xn))
        if bias is not None:
            val = val + bias.astype(np.float64)
            err = err + 4 * U32 * (np.abs(val) + np.abs(bias))
        return val, err

    k, ek = proj(L0["wk"], L0.get("bk"))
    v, ev = proj(L0["wv"], L0.get("bv"))
    D, half = s.head_dim, s.head_dim // 2
    k, ek = k.reshape(s.n_kv_heads, D), ek.reshape(s.n_kv_heads, D)
    if s.qk_norm:
        wn = L0["k_norm"].astype(np.float64)
        ms = np.mean(k * k, axis=1, keepdims=True) + s.rms_eps
        inv = 1.0 / np.sqrt(ms)
        rel = np.sum(np.abs(k) * ek, axis=1, keepdims=True) / (D * ms) + 16 * U32
        k2 = k * inv * wn
        e2 = np.abs(wn) * inv * (ek + np.abs(k) * rel) + 4 * U32 * np.abs(k2)
    else:
        k2, e2 = k, ek
    ang = pos * float(s.rope_theta) ** (-np.arange(half, dtype=np.float64) / half)
    c, sn = np.cos(ang), np.sin(ang)
    a, b = k2[:, :half], k2[:, half:]
    ea, eb = e2[:, :half], e2[:, half:]
    k3 = np.concatenate([a * c - b * sn, a * sn + b * c], axis=1)
    t1 = np.abs(a * c) + np.abs(b * sn)
    t2 = np.abs(a * sn) + np.abs(b * c)
    e3 = np.concatenate([np.abs(c) * ea + np.abs(sn) * eb + 4 * U32 * t1,
                         np.abs(sn) * ea + np.abs(c) * eb + 4 * U32 * t2], axis=1)
    return k3.ravel(), e3.ravel(), v, ev


def layer0_close(got_row, ref_row, val, err, kv_dtype):
    """|gpu - oracle| for layer 0's stored row within the kernel bar; the
    oracle's own row must sit inside the same bound around the double
    recomputation (a check of the bound's arithmetic)."""
    a, b = got_row.astype(np.float64), ref_row.astype(np.float64)
    if kv_dtype == synth.KV_F16:
        tol = err + 2.0 ** -10 * np.maximum(np.abs(a), np.abs(b)) + 2.0 ** -24
    else:
        tol = err + 2 * U32 * np.abs(b)
    assert np.all(np.abs(b - val) <= tol), "bound recomputation disagrees with the oracle"
    bad = np.abs(a - b) > tol
    assert not bad.any(), (np.flatnonzero(bad)[:5], a[bad][:5], b[bad][:5], tol[bad][:5])


def caches_close(dstep, host, kv_dtype, pos, layer0=None):
    for li, (kc, vc) in enumerate(host.caches):
        for which, (dev_c, ref) in enumerate(((dstep.layers[li]["kcache"], kc),
                                              (dstep.layers[li]["vcache"], vc))):
            got = dev_c.cpu().numpy()
            assert np.array_equal(got[:pos], ref[:pos]), "rows before pos must be untouched"
            assert np.array_equal(got[pos + 1:], ref[pos + 1:])
            if li == 0 and layer0 is not None:
                val, err = layer0[2 * which], layer0[2 * which + 1]
                layer0_close(got[pos], ref[pos], val, err, kv_dtype)
                continue
            a, b = got[pos].astype(np.float64), ref[pos].astype(np.float64)
            # one f16 rounding of each side plus the step's named class, taken
            # relative to the row's scale (past layer 0 the f32 path carries the
            # residual stream's rounding, as the logits do)
            rms = np.sqrt(np.mean(b * b))
            tol = np.abs(b) * (2.0 ** -10 if kv_dtype == synth.KV_F16 else 0.0) + STEP_TOL * rms
            bad = np.abs(a - b) > tol
            assert not bad.any(), (li, np.flatnonzero(bad)[:5], a[bad][:5], b[bad][:5])


@functools.lru_cache(maxsize=1)
def weights_for(shape, seed):
    # the 7B-shaped weights take minutes to draw on the host: reused by the
    # tests of one shape
    return synth.step_weights(shape, seed=seed)


def run_case(orc, shape, pos, cap, token=17, steps=1, seed=0):
    w = weights_for(shape, seed)
    caches = [synth.kv_prefix(shape, seed, li, cap, pos) for li in range(shape.n_layers)]
    host = orc.HostStep(w, cap, [(k.copy(), v.copy()) for k, v in caches])
    ds = DeviceStep(w, cap, caches)
    ds.set_state(token, pos)
    tok_ref = token
    rel = []
    for s in range(steps):
        ds.launch()
        torch.cuda.synchronize()
        logits_ref, nxt_ref = host.step(tok_ref, pos + s)
        tok_gpu = int(ds.token.item())
        rel.append(compare_step(ds.logits.cpu().numpy(), logits_ref, tok_gpu, nxt_ref))
        assert int(ds.pos.item()) == pos + s + 1
        assert ds.step.status() == 0
        if tok_gpu != nxt_ref:
            break
        tok_ref = nxt_ref
    if len(rel) == 1:
        caches_close(ds, host, shape.kv_dtype, pos,
                     layer0=layer0_kv_bound(orc, w, shape, token, pos))
    ds.close()
    return rel


def test_step_tiny(orc, q8d):
    rel = run_case(orc, synth.tiny_shape(2), pos=5, cap=16)
    assert rel[0] < STEP_TOL


def test_step_tiny_consecutive_tokens(orc, q8d):
    """Three launches of the same graph decode three consecutive tokens."""
    rel = run_case(orc, synth.tiny_shape(3), pos=0, cap=8, steps=3)
    assert len(rel) == 3


def test_step_launch_host_io(orc, q8d):
    """q8d_step_launch_host: token and position from pinned host memory, the
    next token back to host memory, one call a step.  Three steps decode the
    same tokens as launches with the state set on the device, the oracle's
    tokens, and a mid-sequence restart from the host (a position fed back
    one step) reproduces the step it repeats."""
    shape = synth.tiny_shape(3)
    w = weights_for(shape, 0)
    pos0, cap = 4, 16
    caches = [synth.kv_prefix(shape, 0, li, cap, pos0) for li in range(shape.n_layers)]
    host = orc.HostStep(w, cap, [(k.copy(), v.copy()) for k, v in caches])
    ds = DeviceStep(w, cap, caches)
    h_in = torch.tensor([17, pos0], dtype=torch.int32).pin_memory()
    h_out = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    toks = []
    tok_ref = 17
    for s in range(3):
        h_in[1] = pos0 + s
        ds.launch_host(h_in, h_out)
        torch.cuda.synchronize()
        logits_ref, nxt_ref = host.step(tok_ref, pos0 + s)
        assert compare_step(ds.logits.cpu().numpy(), logits_ref, int(h_out[0]), nxt_ref) < STEP_TOL
        assert int(h_out[0]) == int(ds.token.item())          # the copy is the device token
        assert int(ds.pos.item()) == pos0 + s + 1
        toks.append(int(h_out[0]))
        h_in[0] = int(h_out[0])
        tok_ref = nxt_ref
    # repeat the last step from the host: same input, same position, same token
    h_in[0], h_in[1] = toks[1], pos0 + 2
    ds.launch_host(h_in, h_out)
    torch.cuda.synchronize()
    assert int(h_out[0]) == toks[2]
    # no input copy: continues from the device state
    ds.launch_host(None, h_out)
    torch.cuda.synchronize()
    assert int(ds.pos.item()) == pos0 + 4
    assert ds.step.status() == 0
    ds.close()


def test_step_qwen3_0_6b_shape(orc, q8d):
    run_case(orc, synth.QWEN3_0_6B, pos=511, cap=2048)


def test_step_qwen25_0_5b_shape(orc, q8d):
    run_case(orc, synth.QWEN25_0_5B, pos=511, cap=4096)


def test_step_qwen3_0_6b_ctx2048(orc, q8d):
    """Qwen3-0.6B shape at its stated context 2048: 19 chunks per KV head of
    108 rows, so the attention phase runs two 64-row sub-tiles per chunk."""
    run_case(orc, synth.QWEN3_0_6B, pos=2047, cap=2048)


@pytest.mark.parametrize("pos", [2047, 4095])
def test_step_qwen25_0_5b_contexts(orc, q8d, pos):
    """Qwen2.5-0.5B shape (f32 cache) at its stated contexts 2048 and 4096."""
    run_case(orc, synth.QWEN25_0_5B, pos=pos, cap=4096)


@pytest.mark.slow
def test_step_7b_shape(orc, q8d):
    run_case(orc, synth.QWEN25_7B, pos=2047, cap=2048)


@pytest.mark.slow
def test_step_7b_ctx8192(orc, q8d):
    """7B shape at context 8192: 216-row chunks, four sub-tiles each."""
    run_case(orc, synth.QWEN25_7B, pos=8191, cap=8192)


# Chunks longer than the attention phase's sub-tile (64 rows; 32 for
# head_dim 128 with an f32 cache) for every (head_dim, cache type) instance
# of the step kernel: with 152 CTAs and 8 KV heads a chunk is
# ceil(L / 19) rows.  The last case (4 KV heads: 38 chunks of 17 rows at
# L = 620) leaves the last chunk empty.
SUBTILE_CASES = [
    ("d128-f16", 128, synth.KV_F16, 8, 2999, True, False),
    ("d128-f32", 128, synth.KV_F32, 8, 1000, False, True),
    ("d64-f16", 64, synth.KV_F16, 8, 2999, False, True),
    ("d64-f32", 64, synth.KV_F32, 8, 2999, True, False),
    ("d128-f16-empty-chunk", 128, synth.KV_F16, 4, 619, True, True),
]


@pytest.mark.parametrize("name,D,kvd,Hk,pos,qkn,bias", SUBTILE_CASES)
def test_step_attention_subtiles(orc, q8d, name, D, kvd, Hk, pos, qkn, bias):
    shape = synth.ModelShape(name, 256, 2, 2 * Hk, Hk, D, 512, 500,
                             qk_norm=qkn, qkv_bias=bias, kv_dtype=kvd)
    run_case(orc, shape, pos=pos, cap=pos + 64)


# The largest query groups per KV head the step takes: 12 with an f16 cache
# (the tensor-core attention prepares one q row per warp beside its 8 pair
# warps), 16 with an f32 cache (one head per warp).
GROUP_CASES = [
    ("g12-d64-f16", 64, synth.KV_F16, 12),
    ("g12-d128-f16", 128, synth.KV_F16, 12),
    ("g16-d128-f32", 128, synth.KV_F32, 16),
    ("g16-d64-f32", 64, synth.KV_F32, 16),
]


@pytest.mark.parametrize("name,D,kvd,G", GROUP_CASES)
def test_step_large_query_groups(orc, q8d, name, D, kvd, G):
    shape = synth.ModelShape(name, 256, 2, G, 1, D, 512, 500,
                             qk_norm=True, qkv_bias=True, kv_dtype=kvd)
    run_case(orc, shape, pos=300, cap=512)


def test_step_head_dim_128_f32_cache(orc, q8d):
    # the step kernel's (head_dim 128, f32 cache) instance
    shape = synth.ModelShape("d128-f32", 256, 2, 4, 2, 128, 320, 600,
                             qk_norm=True, qkv_bias=False, kv_dtype=synth.KV_F32)
    run_case(orc, shape, pos=77, cap=256)


def test_step_odd_block_counts(orc, q8d):
    # rows of 33 and 35 blocks: paired warps whose block alignment changes
    # from row to row (hidden 1056, ffn 1120), q width 256 (8 blocks)
    shape = synth.ModelShape("odd-blocks", 1056, 2, 4, 2, 64, 1120, 700,
                             qk_norm=False, qkv_bias=True, kv_dtype=synth.KV_F16)
    run_case(orc, shape, pos=300, cap=512)


def test_step_tensor_core_phases_ragged_sets(orc, q8d):
    # every matvec phase on the tensor-core path (n % 256 == 0, >= 64
    # blocks a row: hidden 2048, ffn 2560): CTA row ranges of 17 (q|k|v,
    # gate|up), 14 (o), 20 (lm_head of 3001 rows) rows, so tiles of 8 rows
    # end in partial ones, and some straddle the q / k / v boundaries
    shape = synth.ModelShape("tc-ragged", 2048, 2, 16, 2, 128, 2560, 3001,
                             qk_norm=False, qkv_bias=True, kv_dtype=synth.KV_F16)
    run_case(orc, shape, pos=700, cap=1024)


def test_step_position_past_cache_flags_error(orc, q8d):
    shape = synth.tiny_shape(1)
    w = synth.step_weights(shape, seed=1)
    ds = DeviceStep(w, 4)
    ds.set_state(3, 4)          # pos == cap
    ds.launch()
    torch.cuda.synchronize()
    err = ds.step.status()
    assert err & q8d.Q8D_DERR_LEN_RANGE
    assert np.isnan(ds.logits.cpu().numpy()).all()
    ds.close()


def test_step_refuses_more_kv_heads_than_sms(q8d):
    """The attention phase gives each KV head at least one CTA of the
    one-per-SM grid: more KV heads than SMs are refused at creation."""
    hk = torch.cuda.get_device_properties(0).multi_processor_count + 8
    shape = synth.ModelShape("many-kv", 256, 1, hk, hk, 64, 256, 100,
                             qk_norm=False, qkv_bias=False, kv_dtype=synth.KV_F16)
    w = synth.step_weights(shape, seed=1)
    with pytest.raises(q8d.Q8DError) as e:
        DeviceStep(w, 4)
    assert e.value.status == q8d.Q8D_EUNSUPPORTED


def test_step_bad_token_flags_error(orc, q8d):
    shape = synth.tiny_shape(1)
    w = synth.step_weights(shape, seed=1)
    ds = DeviceStep(w, 4)
    ds.set_state(shape.vocab + 5, 0)
    ds.launch()
    torch.cuda.synchronize()
    assert ds.step.status() & q8d.Q8D_DERR_TOKEN_RANGE
    ds.close()


def test_step_kernel_count(orc, q8d):
    shape = synth.tiny_shape(2)
    ds = DeviceStep(synth.step_weights(shape), 4)
    # the whole step is one persistent kernel (embedding, every layer's
    # phases, lm_head and argmax); the graph's other node is a memset
    assert ds.kernel_count() == 1
    ds.close()


def test_step_wait_limit_expiry_leaves_context_usable(orc, q8d):
    """A grid-barrier wait limit of one poll makes the step give up at a
    barrier (no CTA waits for an arrival that is withheld forever: every
    wait is bounded); the step must return, set Q8D_DERR_WAIT, leave the
    position unadvanced, and the next step with the default limit must
    match the oracle."""
    shape = synth.tiny_shape(2)
    w = weights_for(shape, 0)
    cap, pos = 16, 5
    caches = [synth.kv_prefix(shape, 0, li, cap, pos) for li in range(shape.n_layers)]
    host = orc.HostStep(w, cap, [(k.copy(), v.copy()) for k, v in caches])
    ds = DeviceStep(w, cap, caches)
    ds.step.set_wait_limit(1)
    ds.set_state(17, pos)
    ds.launch()
    torch.cuda.synchronize()
    err = ds.step.status()
    assert err & q8d.Q8D_DERR_WAIT, err
    assert int(ds.pos.item()) == pos, "an abandoned step must not advance the position"
    ds.step.set_wait_limit(0)   # back to the default (about a second)
    ds.err.zero_()
    ds.set_state(17, pos)
    ds.launch()
    torch.cuda.synchronize()
    assert ds.step.status() == 0
    logits_ref, nxt = host.step(17, pos)
    compare_step(ds.logits.cpu().numpy(), logits_ref, int(ds.token.item()), nxt)
    assert int(ds.pos.item()) == pos + 1
    ds.close()
