"""Seeded synthetic inputs for the Q8_0 decode path.

This module only draws random numbers and lays them out in the formats the
path reads (Q8_0 blocks, f32/f16 arrays).  It holds none of the method's
arithmetic.  Both the oracle-side tests and the CUDA-side tests/bench take
their inputs from here; nothing here imports the oracle or the CUDA library.

Distributions (stated once, used everywhere):
  * activations, queries, K/V: N(0, 1), drawn in double, rounded to f32
    (K/V for an f16 cache rounded to f16 by numpy's float16 cast),
  * Q8_0 quants: integers uniform on [-127, 127],
  * Q8_0 scales: uniform on [1e-3, 2e-2], rounded to f16 (all normal halves),
  * RMSNorm gains: 1 + 0.1 N(0, 1); biases: 0.1 N(0, 1).
Every tensor has its own stream: numpy's PCG64 seeded by the pair
(workload seed, crc32 of the tensor's name).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

QBLOCK = 32          # quants per Q8_0 block
QBLOCK_BYTES = 34    # 2-byte little-endian f16 scale + 32 int8 quants

KV_F32 = 0
KV_F16 = 1
KV_Q8_0 = 2  # packed cache: rows of kv_width/32 Q8_0 blocks


def stream(seed: int, name: str) -> np.random.Generator:
    """Independent generator for one named tensor of one seeded workload."""
    return np.random.default_rng([int(seed) & 0xFFFFFFFF, zlib.crc32(name.encode())])


def normal_f32(seed: int, name: str, shape) -> np.ndarray:
    return stream(seed, name).standard_normal(shape).astype(np.float32)


def normal_f16(seed: int, name: str, shape) -> np.ndarray:
    return stream(seed, name).standard_normal(shape).astype(np.float16)


def gains(seed: int, name: str, n: int) -> np.ndarray:
    return (1.0 + 0.1 * stream(seed, name).standard_normal(n)).astype(np.float32)


def biases(seed: int, name: str, n: int) -> np.ndarray:
    return (0.1 * stream(seed, name).standard_normal(n)).astype(np.float32)


def pack_q8(scales_f16: np.ndarray, quants_i8: np.ndarray) -> np.ndarray:
    """Lay out Q8_0 blocks: scales [p, n/32] (float16), quants [p, n/32, 32]
    (int8) -> uint8 [p, n/32 * 34], each block = LE f16 scale then 32 quants."""
    p, bpr = scales_f16.shape
    out = np.empty((p, bpr, QBLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(scales_f16.astype("<f2")).view(np.uint8).reshape(p, bpr, 2)
    out[:, :, 2:] = quants_i8.view(np.uint8)
    return out.reshape(p, bpr * QBLOCK_BYTES)


def q8_matrix(seed: int, name: str, p: int, n: int, scale_lo: float = 1e-3,
              scale_hi: float = 2e-2) -> np.ndarray:
    """Random [p][n] Q8_0 matrix as uint8 [p, n/32*34]."""
    if n % QBLOCK:
        raise ValueError("n must be a multiple of 32")
    g = stream(seed, name)
    bpr = n // QBLOCK
    quants = g.integers(-127, 128, size=(p, bpr, QBLOCK), dtype=np.int8)
    scales = g.uniform(scale_lo, scale_hi, size=(p, bpr)).astype(np.float16)
    return pack_q8(scales, quants)


def q8_const_matrix(p: int, n: int, scale_bits: int, quant: int) -> np.ndarray:
    """Every block has the same scale bit pattern and every quant the same value."""
    bpr = n // QBLOCK
    scales = np.full((p, bpr), scale_bits, dtype=np.uint16).view(np.float16)
    quants = np.full((p, bpr, QBLOCK), quant, dtype=np.int8)
    return pack_q8(scales, quants)


def q8_from_parts(seed: int, name: str, p: int, n: int, scale_bits: int) -> np.ndarray:
    """Random quants in [-127, 127] with every scale set to one bit pattern."""
    g = stream(seed, name)
    bpr = n // QBLOCK
    quants = g.integers(-127, 128, size=(p, bpr, QBLOCK), dtype=np.int8)
    scales = np.full((p, bpr), scale_bits, dtype=np.uint16).view(np.float16)
    return pack_q8(scales, quants)


class PagesLCG:
    """The tiny deterministic generator of the pages' GPU kernel tests
    ("IV.4: One command buffer per token", "The correctness ladder"):
    a 64-bit LCG whose top bits map to [-1, 1)."""

    MUL = 6364136223846793005
    INC = 1442695040888963407

    def __init__(self, seed: int):
        self.state = seed & 0xFFFFFFFFFFFFFFFF

    def next_f32(self) -> np.float32:
        self.state = (self.state * self.MUL + self.INC) & 0xFFFFFFFFFFFFFFFF
        return np.float32(np.float32(self.state >> 33) / np.float32(1 << 31) - np.float32(1.0))


def pages_fabricated_q8(p: int, n: int, seed: int) -> np.ndarray:
    """The pages' Q8 weight fabricator: every block's scale bytes are
    (0x00, 0x2c) and each quant is the LCG draw times 127, truncated to int8."""
    g = PagesLCG(seed)
    bpr = n // QBLOCK
    out = np.empty((p * bpr, QBLOCK_BYTES), dtype=np.uint8)
    for b in range(p * bpr):
        out[b, 0] = 0x00
        out[b, 1] = 0x2C
        for j in range(QBLOCK):
            out[b, 2 + j] = np.int8(int(g.next_f32() * np.float32(127.0))).view(np.uint8)
    return out.reshape(p, bpr * QBLOCK_BYTES)


# ---------------------------------------------------------------------------
# Model shapes of the synthetic decode-step workloads (the pages' Qwen3-0.6B
# and Qwen2.5 models; no trained weights are used anywhere).
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class ModelShape:
    name: str
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    qk_norm: bool
    qkv_bias: bool
    kv_dtype: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    def matvec_shapes(self):
        """(name, n, p) of every Q8_0 matvec of one step, in step order."""
        h, q, kv, f = self.hidden, self.q_width, self.kv_width, self.ffn
        per = [("wq", h, q), ("wk", h, kv), ("wv", h, kv), ("wo", q, h),
               ("wg", h, f), ("wu", h, f), ("wd", f, h)]
        out = []
        for li in range(self.n_layers):
            out += [(f"l{li}.{nm}", n, p) for nm, n, p in per]
        out.append(("lm_head", h, self.vocab))
        return out

    def weight_bytes(self) -> int:
        return sum(p * (n // QBLOCK) * QBLOCK_BYTES for _, n, p in self.matvec_shapes())


QWEN3_0_6B = ModelShape("qwen3-0.6b", 1024, 28, 16, 8, 128, 3072, 151936,
                        qk_norm=True, qkv_bias=False, kv_dtype=KV_F16)
QWEN25_0_5B = ModelShape("qwen2.5-0.5b", 896, 24, 14, 2, 64, 4864, 151936,
                         qk_norm=False, qkv_bias=True, kv_dtype=KV_F32)
QWEN25_7B = ModelShape("qwen2.5-7b", 3584, 28, 28, 4, 128, 18944, 152064,
                       qk_norm=False, qkv_bias=True, kv_dtype=KV_F16)

MODELS = {m.name: m for m in (QWEN3_0_6B, QWEN25_0_5B, QWEN25_7B)}


def tiny_shape(n_layers: int = 2) -> ModelShape:
    """A small step of the same structure for fast tests: hidden 192 (6
    blocks), ffn 352 (11 blocks, so down-projection rows are only 2-byte
    aligned), head_dim 64, GQA group 3, both QK-norm and q/k/v biases."""
    return ModelShape("tiny", 192, n_layers, 6, 2, 64, 352, 1000,
                      qk_norm=True, qkv_bias=True, kv_dtype=KV_F16)


@dataclass
class StepWeights:
    """Host copies of every tensor of a synthetic decode-step model."""
    shape: ModelShape
    layers: list
    embed: np.ndarray
    out_norm: np.ndarray
    lm_head: np.ndarray


def step_weights(shape: ModelShape, seed: int = 0) -> StepWeights:
    """Draws every tensor (matrices in parallel threads; each has its own
    stream, so the values do not depend on the thread count)."""
    import concurrent.futures as cf
    import os
    s = shape
    jobs = {}
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        for li in range(s.n_layers):
            for nm, n, p in [("wq", s.hidden, s.q_width), ("wk", s.hidden, s.kv_width),
                             ("wv", s.hidden, s.kv_width), ("wo", s.q_width, s.hidden),
                             ("wg", s.hidden, s.ffn), ("wu", s.hidden, s.ffn),
                             ("wd", s.ffn, s.hidden)]:
                jobs[(li, nm)] = ex.submit(q8_matrix, seed, f"l{li}.{nm}", p, n)
        fe = ex.submit(q8_matrix, seed, "embed", s.vocab, s.hidden)
        fl = ex.submit(q8_matrix, seed, "lm_head", s.vocab, s.hidden)
        mats = {k: f.result() for k, f in jobs.items()}
        embed, lm_head = fe.result(), fl.result()
    layers = []
    for li in range(s.n_layers):
        L = {}
        for nm in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
            L[nm] = mats[(li, nm)]
        L["attn_norm"] = gains(seed, f"l{li}.attn_norm", s.hidden)
        L["ffn_norm"] = gains(seed, f"l{li}.ffn_norm", s.hidden)
        if s.qk_norm:
            L["q_norm"] = gains(seed, f"l{li}.q_norm", s.head_dim)
            L["k_norm"] = gains(seed, f"l{li}.k_norm", s.head_dim)
        if s.qkv_bias:
            L["bq"] = biases(seed, f"l{li}.bq", s.q_width)
            L["bk"] = biases(seed, f"l{li}.bk", s.kv_width)
            L["bv"] = biases(seed, f"l{li}.bv", s.kv_width)
        layers.append(L)
    return StepWeights(s, layers, embed=embed, out_norm=gains(seed, "out_norm", s.hidden),
                       lm_head=lm_head)


def q8_kv_cache(seed: int, name: str, cap: int, kv_width: int, rows: int | None = None):
    """A packed Q8_0 cache [cap, kv_width/32*34] (uint8) whose first `rows`
    rows (all if None) hold random blocks: quants uniform on [-127, 127],
    scales uniform on [4e-3, 3e-2] (the range of N(0, 1) rows' blocks);
    the other rows are zero."""
    rows = cap if rows is None else rows
    out = np.zeros((cap, kv_width // QBLOCK * QBLOCK_BYTES), dtype=np.uint8)
    if rows > 0:
        out[:rows] = q8_matrix(seed, name, rows, kv_width, 4e-3, 3e-2)
    return out


def kv_prefix(shape: ModelShape, seed: int, layer: int, cap: int, rows: int):
    """Cache contents for `rows` already-decoded positions: N(0,1) in the cache
    dtype; rows past `rows` are zero.  Returns (kcache, vcache) arrays
    [cap, kv_width] of float16 or float32."""
    if shape.kv_dtype == KV_Q8_0:
        return (q8_kv_cache(seed, f"l{layer}.kprefix", cap, shape.kv_width, rows),
                q8_kv_cache(seed, f"l{layer}.vprefix", cap, shape.kv_width, rows))
    dt = np.float16 if shape.kv_dtype == KV_F16 else np.float32
    kc = np.zeros((cap, shape.kv_width), dtype=dt)
    vc = np.zeros((cap, shape.kv_width), dtype=dt)
    if rows > 0:
        kc[:rows] = stream(seed, f"l{layer}.kprefix").standard_normal((rows, shape.kv_width)).astype(dt)
        vc[:rows] = stream(seed, f"l{layer}.vprefix").standard_normal((rows, shape.kv_width)).astype(dt)
    return kc, vc


# ---------------------------------------------------------------------------
# Device-side generation (same distributions, torch's generator) for
# workloads too large to draw on the host in reasonable time.  Values differ
# from the numpy streams above; they are used where no oracle comparison of
# the exact values is made (throughput runs).
# ---------------------------------------------------------------------------

def _torch_gen(seed: int, name: str, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(((int(seed) & 0xFFFFFFFF) << 32) ^ zlib.crc32(name.encode()))
    return g


def q8_matrix_torch(seed: int, name: str, p: int, n: int, device="cuda", scale_lo: float = 1e-3,
                    scale_hi: float = 2e-2):
    import torch
    g = _torch_gen(seed, name, device)
    bpr = n // QBLOCK
    out = torch.empty((p, bpr, QBLOCK_BYTES), dtype=torch.uint8, device=device)
    q = torch.randint(-127, 128, (p, bpr, QBLOCK), dtype=torch.int8, device=device, generator=g)
    out[:, :, 2:] = q.view(torch.uint8)
    del q
    s = torch.rand((p, bpr), dtype=torch.float32, device=device, generator=g)
    s = (s * (scale_hi - scale_lo) + scale_lo).to(torch.float16)
    out[:, :, 0:2] = s.view(torch.uint8).view(p, bpr, 2)
    return out.view(p, bpr * QBLOCK_BYTES)


def normal_torch(seed: int, name: str, shape, dtype, device="cuda"):
    import torch
    g = _torch_gen(seed, name, device)
    return torch.randn(shape, dtype=torch.float32, device=device, generator=g).to(dtype)


class TorchStepWeights:
    """Same fields as StepWeights, holding device tensors drawn on the GPU."""

    def __init__(self, shape: ModelShape, seed: int = 0, device="cuda"):
        import torch
        s = shape
        self.shape = s
        self.layers = []
        for li in range(s.n_layers):
            L = {}
            for nm, n, p in [("wq", s.hidden, s.q_width), ("wk", s.hidden, s.kv_width),
                             ("wv", s.hidden, s.kv_width), ("wo", s.q_width, s.hidden),
                             ("wg", s.hidden, s.ffn), ("wu", s.hidden, s.ffn),
                             ("wd", s.ffn, s.hidden)]:
                L[nm] = q8_matrix_torch(seed, f"l{li}.{nm}", p, n, device)
            for nm, n in [("attn_norm", s.hidden), ("ffn_norm", s.hidden)]:
                L[nm] = 1.0 + 0.1 * normal_torch(seed, f"l{li}.{nm}", n, torch.float32, device)
            if s.qk_norm:
                for nm in ("q_norm", "k_norm"):
                    L[nm] = 1.0 + 0.1 * normal_torch(seed, f"l{li}.{nm}", s.head_dim, torch.float32, device)
            if s.qkv_bias:
                for nm, n in [("bq", s.q_width), ("bk", s.kv_width), ("bv", s.kv_width)]:
                    L[nm] = 0.1 * normal_torch(seed, f"l{li}.{nm}", n, torch.float32, device)
            self.layers.append(L)
        self.embed = q8_matrix_torch(seed, "embed", s.vocab, s.hidden, device)
        self.out_norm = 1.0 + 0.1 * normal_torch(seed, "out_norm", s.hidden, torch.float32, device)
        self.lm_head = q8_matrix_torch(seed, "lm_head", s.vocab, s.hidden, device)
