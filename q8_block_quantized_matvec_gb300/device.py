"""Device-resident decode-step model: uploads host weight arrays once
(as the pages' decoder does at start-up) and builds the q8d_step_desc.

PyTorch is used only to own device memory; all compute is libq8d's."""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import LayerDesc, Step, StepDesc, Q8D_KV_F16


def to_device(a, device="cuda") -> torch.Tensor:
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceStep:
    """Holds device copies of a model's tensors, its KV caches and the
    captured step.  `weights` exposes .shape (dims), .layers (list of dicts
    of numpy arrays), .embed, .out_norm, .lm_head."""

    def __init__(self, weights, cap: int, caches=None, device="cuda", stream=None,
                 keep_logits=True):
        s = weights.shape
        self.shape = s
        self.cap = cap
        self.device = device
        dt = torch.float16 if s.kv_dtype == Q8D_KV_F16 else torch.float32
        self.layers = []
        for li, L in enumerate(weights.layers):
            d = {k: to_device(v, device) for k, v in L.items()}
            if caches is not None:
                d["kcache"] = to_device(caches[li][0], device)
                d["vcache"] = to_device(caches[li][1], device)
            else:
                d["kcache"] = torch.zeros((cap, s.kv_width), dtype=dt, device=device)
                d["vcache"] = torch.zeros((cap, s.kv_width), dtype=dt, device=device)
            self.layers.append(d)
        self.embed = to_device(weights.embed, device)
        self.out_norm = to_device(weights.out_norm, device)
        self.lm_head = to_device(weights.lm_head, device)
        # token id and position side by side: one 8-byte copy sets both
        self.token_pos = torch.zeros(2, dtype=torch.int32, device=device)
        self.token = self.token_pos[0:1]
        self.pos = self.token_pos[1:2]
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.logits = torch.empty(s.vocab, dtype=torch.float32, device=device) if keep_logits else None

        arr = (LayerDesc * s.n_layers)()
        for li, d in enumerate(self.layers):
            ld = arr[li]
            for nm in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "attn_norm", "ffn_norm",
                       "kcache", "vcache"):
                setattr(ld, nm, d[nm].data_ptr())
            for nm in ("q_norm", "k_norm", "bq", "bk", "bv"):
                setattr(ld, nm, d[nm].data_ptr() if nm in d else None)
        self._arr = arr
        desc = StepDesc(s.hidden, s.n_layers, s.n_heads, s.n_kv_heads, s.head_dim, s.ffn, s.vocab,
                        int(s.qk_norm), int(s.qkv_bias), s.kv_dtype, cap, s.rms_eps, s.rope_theta,
                        self.embed.data_ptr(), self.out_norm.data_ptr(), self.lm_head.data_ptr(),
                        C.cast(arr, C.POINTER(LayerDesc)), self.token.data_ptr(),
                        self.pos.data_ptr(), self.err.data_ptr(),
                        self.logits.data_ptr() if self.logits is not None else None)
        self.desc = desc
        self.step = Step(desc, arr, stream)

    def set_state(self, token: int, pos: int):
        self.token.fill_(int(token))
        self.pos.fill_(int(pos))

    def launch(self, stream=None):
        self.step.launch(stream)

    def launch_host(self, h_token_pos, h_next_token, stream=None):
        """One step with host I/O (q8d_step_launch_host): pinned int32
        [token, position] in, pinned int32 [1] next token out."""
        self.step.launch_host(h_token_pos, h_next_token, stream)

    def kernel_count(self) -> int:
        return self.step.kernel_count()

    def close(self):
        self.step.close()
