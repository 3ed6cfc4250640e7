"""Move seeded host inputs onto the GPU as torch tensors, and back.

Only marshalling happens here: bf16 values travel as their raw 16-bit
patterns. The tests, the benchmark and the smoke check use these helpers to
drive libmla through its C ABI.
"""
from __future__ import annotations

import numpy as np

from . import _lib
from .synth import Workload


def to_device(storage, dtype, device="cuda"):
    import torch
    if dtype == "f32" or storage.dtype == np.float32:
        return torch.from_numpy(np.ascontiguousarray(storage)).to(device)
    if storage.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(storage).view(np.int16)).to(device)
        return t.view(torch.bfloat16)
    if storage.dtype == np.int32:
        return torch.from_numpy(np.ascontiguousarray(storage)).to(device)
    raise TypeError(storage.dtype)


def to_host_f32(t):
    """Device tensor (fp32 or bf16) -> numpy float32 with the exact values."""
    import torch
    if t.dtype == torch.bfloat16:
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32)
    return t.float().cpu().numpy()


def config_for(w: Workload, impl=_lib.MLA_IMPL_AUTO):
    return _lib.make_config(w.n_h, w.d_model, w.d_c, w.d_r, w.d_nope, w.d_v,
                            block_size=w.block_size, rope_base=w.rope_base,
                            softmax_scale=0.0, dtype=w.dtype, impl=impl)


class DeviceWeights:
    """Weights uploaded and absorbed (mla_absorb_weights)."""

    def __init__(self, w: Workload, wts, cfg, stream=None):
        import torch
        self.raw = {k: to_device(v, w.dtype) for k, v in wts.raw.items()
                    if k in ("W_dkv", "W_kr", "W_uk", "W_uv")}
        self.handle = _lib.mla_absorb_weights(cfg, self.raw["W_dkv"], self.raw["W_kr"],
                                              self.raw["W_uk"], self.raw["W_uv"], stream)
        torch.cuda.synchronize()

    def free(self):
        if self.handle is not None:
            _lib.mla_weights_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass
