"""q8d_gqa_decode_attn_noalloc: the decode attention for callers that cannot
allocate device memory (their memory belongs to a host framework's
allocator, or they cannot afford cudaMalloc's device-wide synchronisation).
It keeps its split-K scratch in a fixed array inside the library.  Checked
through the C ABI against q8d_gqa_decode_attn with a caller workspace, on
two calls in a row (the array keeps the previous call's contents).  This
file is collected last on purpose."""
import ctypes as C
import math

import numpy as np
import pytest
import torch

import synth
from conftest import dev

pytestmark = pytest.mark.gpu
TOL = 1e-5


def _inputs(seed, H, Hk, D, cap, lens, dtype):
    kvw = Hk * D
    batch = len(lens)
    mk = synth.normal_f16 if dtype == synth.KV_F16 else synth.normal_f32
    kc = mk(seed, "na.k", (batch, cap, kvw))
    vc = mk(seed, "na.v", (batch, cap, kvw))
    q = synth.normal_f32(seed, "na.q", (batch, H * D))
    return q, kc, vc


def _run_pair(q8d, q, kc, vc, dtype, H, Hk, D, cap, lens):
    L = q8d.lib()
    batch = len(lens)
    stride = cap * Hk * D
    qd, kcd, vcd = dev(q), dev(kc), dev(vc)
    d_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = torch.full((batch, H * D), float("nan"), device="cuda")
    got = torch.full((batch, H * D), float("nan"), device="cuda")
    wsb = q8d.q8d_gqa_workspace_bytes(batch, H, Hk, D, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    scale = 1 / math.sqrt(D)
    rc = L.q8d_gqa_decode_attn(qd.data_ptr(), None, None, kcd.data_ptr(), vcd.data_ptr(), dtype,
                               ref.data_ptr(), batch, H, Hk, D, cap, stride, d_lens.data_ptr(),
                               C.c_float(scale), ws.data_ptr(), wsb, err.data_ptr(), s)
    assert rc == 0
    rc = L.q8d_gqa_decode_attn_noalloc(qd.data_ptr(), None, None, kcd.data_ptr(), vcd.data_ptr(),
                                       dtype, got.data_ptr(), batch, H, Hk, D, cap, stride,
                                       d_lens.data_ptr(), C.c_float(scale), err.data_ptr(), s)
    assert rc == 0, q8d.strerror(rc)
    torch.cuda.synchronize()
    assert err.item() == 0
    return got.cpu().numpy(), ref.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice(q8d, orc):
    # two different calls in a row: the second must not see the first's scratch
    cases = [(28, 4, 128, synth.KV_F16, 4096, [4096, 1, 2049]),
             (14, 2, 64, synth.KV_F32, 700, [513])]
    for seed, (H, Hk, D, dtype, cap, lens) in enumerate(cases):
        q, kc, vc = _inputs(seed, H, Hk, D, cap, lens, dtype)
        got, ref = _run_pair(q8d, q, kc, vc, dtype, H, Hk, D, cap, lens)
        for b, Lb in enumerate(lens):
            oref, ab = orc.gqa_decode_attn(q[b], kc[b], vc[b], dtype, H, Hk, D, Lb, 1 / math.sqrt(D))
            assert np.all(np.abs(got[b] - ref[b]) <= 2 * TOL * ab)
            assert np.all(np.abs(got[b] - oref) <= TOL * ab)


def test_noalloc_refuses_oversized_scratch(q8d):
    L = q8d.lib()
    limit = L.q8d_noalloc_scratch_bytes()
    # many sequences of many heads need more scratch than the fixed array holds
    batch, H, Hk, D, cap = 64, 64, 4, 128, 65536
    assert q8d.q8d_gqa_workspace_bytes(batch, H, Hk, D, cap) > limit
    rc = L.q8d_gqa_decode_attn_noalloc(0x10000, None, None, 0x20000, 0x30000, 1, 0x40000, batch,
                                       H, Hk, D, cap, cap * Hk * D, 0x50000, C.c_float(0.1),
                                       0x60000, None)
    assert rc == q8d.Q8D_ERANGE
