"""Device-resident expert sets: packed weight buffers and pointer tables.

Holds the E packed experts of one layer in two device allocations (codes and
scales, one fixed-size slot per expert) plus the two device arrays of expert
pointers that a moe_expert_table refers to.  torch provides the memory; the
re-layout itself is moe_ffn_pack_expert.
"""
from __future__ import annotations

import torch

from . import (config, expert_table, moe_ffn_packed_codes_bytes, moe_ffn_packed_scales_bytes,
               moe_ffn_pack_expert)


class ExpertSet:
    def __init__(self, handle, cfg, num_experts: int | None = None, device: int = 0):
        self.handle = handle
        self.cfg = cfg
        self.E = cfg.num_experts if num_experts is None else num_experts
        self.code_bytes = moe_ffn_packed_codes_bytes(cfg)
        self.scale_bytes = moe_ffn_packed_scales_bytes(cfg)
        dev = torch.device("cuda", device)
        # slots padded to 256 bytes so every expert starts aligned
        self.code_stride = (self.code_bytes + 255) // 256 * 256
        self.scale_stride = (self.scale_bytes + 255) // 256 * 256
        self.codes = torch.empty(self.E * self.code_stride, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(self.E * self.scale_stride, dtype=torch.uint8, device=dev)
        cb, sb = self.codes.data_ptr(), self.scales.data_ptr()
        self.code_ptrs = torch.tensor([cb + e * self.code_stride for e in range(self.E)],
                                      dtype=torch.int64, device=dev)
        self.scale_ptrs = torch.tensor([sb + e * self.scale_stride for e in range(self.E)],
                                       dtype=torch.int64, device=dev)
        self.table = expert_table(self.code_ptrs, self.scale_ptrs)

    def code_slot(self, e: int) -> int:
        return self.codes.data_ptr() + e * self.code_stride

    def scale_slot(self, e: int) -> int:
        return self.scales.data_ptr() + e * self.scale_stride

    def load(self, e: int, canon_codes, canon_scales, stream=None) -> None:
        """Pack one expert from the published layout (device buffers)."""
        moe_ffn_pack_expert(self.handle, canon_codes, canon_scales, self.code_slot(e),
                            self.scale_slot(e), stream)

    def bytes(self) -> int:
        return self.E * (self.code_bytes + self.scale_bytes)


__all__ = ["ExpertSet", "config"]
