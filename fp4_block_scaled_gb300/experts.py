"""Device-resident expert sets: packed expert blobs and their pointer table.

Holds the E packed experts of one layer in one device allocation (one
fixed-size slot per expert, 256-byte aligned) plus the device array of expert
pointers that a moe_expert_table refers to.  torch provides the memory; the
re-layout itself is moe_ffn_pack_expert.
"""
from __future__ import annotations

import torch

from . import config, expert_table, moe_ffn_packed_expert_bytes, moe_ffn_pack_expert


class ExpertSet:
    def __init__(self, handle, cfg, num_experts: int | None = None, device: int = 0):
        self.handle = handle
        self.cfg = cfg
        self.E = cfg.num_experts if num_experts is None else num_experts
        self.blob_bytes = moe_ffn_packed_expert_bytes(cfg)
        dev = torch.device("cuda", device)
        # slots padded to 256 bytes so every expert starts aligned
        self.stride = (self.blob_bytes + 255) // 256 * 256
        self.blobs = torch.empty(self.E * self.stride, dtype=torch.uint8, device=dev)
        base = self.blobs.data_ptr()
        self.ptrs = torch.tensor([base + e * self.stride for e in range(self.E)], dtype=torch.int64, device=dev)
        self.table = expert_table(self.ptrs)

    def slot(self, e: int) -> int:
        return self.blobs.data_ptr() + e * self.stride

    def load(self, e: int, canon_codes, canon_scales, stream=None) -> None:
        """Pack one expert from the published layout (device buffers)."""
        moe_ffn_pack_expert(self.handle, canon_codes, canon_scales, self.slot(e), stream)

    def bytes(self) -> int:
        return self.E * self.blob_bytes


__all__ = ["ExpertSet", "config"]
