"""The captured decode step (q8d_step_*) against the oracle's double-precision
step.  Named tolerance class for a whole step (28 layers of f32 against f64):
|logit_gpu - logit_oracle| <= 1e-3 * max|logit_oracle|; the argmax must
agree unless the oracle's top-2 gap is inside that bound; appended KV rows
agree to one f16 rounding step."""
import numpy as np
import pytest
import torch

import synth
from q8_block_quantized_matvec_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu
STEP_TOL = 1e-3


def compare_step(logits_gpu, logits_ref, tok_gpu, tok_ref):
    scale = np.max(np.abs(logits_ref))
    err = np.max(np.abs(logits_gpu.astype(np.float64) - logits_ref))
    assert err <= STEP_TOL * scale, (err, scale)
    if tok_gpu != tok_ref:
        top = np.sort(logits_ref.astype(np.float64))[-2:]
        assert top[1] - top[0] <= 2 * STEP_TOL * scale, "argmax differs on a clear winner"
    return err / scale


def caches_close(dstep, host, kv_dtype, pos):
    for li, (kc, vc) in enumerate(host.caches):
        for dev_c, ref in ((dstep.layers[li]["kcache"], kc), (dstep.layers[li]["vcache"], vc)):
            got = dev_c.cpu().numpy()
            assert np.array_equal(got[:pos], ref[:pos]), "rows before pos must be untouched"
            a, b = got[pos].astype(np.float64), ref[pos].astype(np.float64)
            # one f16 rounding of each side plus the step's named class, taken
            # relative to the row's scale (past layer 0 the f32 path carries the
            # residual stream's rounding, as the logits do)
            rms = np.sqrt(np.mean(b * b))
            tol = np.abs(b) * (2.0 ** -10 if kv_dtype == synth.KV_F16 else 0.0) + STEP_TOL * rms
            bad = np.abs(a - b) > tol
            assert not bad.any(), (li, np.flatnonzero(bad)[:5], a[bad][:5], b[bad][:5])
            assert np.array_equal(got[pos + 1:], ref[pos + 1:])


def run_case(orc, shape, pos, cap, token=17, steps=1, seed=0):
    w = synth.step_weights(shape, seed=seed)
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
    caches_close(ds, host, shape.kv_dtype, pos + len(rel) - 1) if len(rel) == 1 else None
    ds.close()
    return rel


def test_step_tiny(orc, q8d):
    rel = run_case(orc, synth.tiny_shape(2), pos=5, cap=16)
    assert rel[0] < STEP_TOL


def test_step_tiny_consecutive_tokens(orc, q8d):
    """Three launches of the same graph decode three consecutive tokens."""
    rel = run_case(orc, synth.tiny_shape(3), pos=0, cap=8, steps=3)
    assert len(rel) == 3


def test_step_qwen3_0_6b_shape(orc, q8d):
    run_case(orc, synth.QWEN3_0_6B, pos=511, cap=2048)


def test_step_qwen25_0_5b_shape(orc, q8d):
    run_case(orc, synth.QWEN25_0_5B, pos=511, cap=4096)


@pytest.mark.slow
def test_step_7b_shape(orc, q8d):
    run_case(orc, synth.QWEN25_7B, pos=2047, cap=2048)


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
