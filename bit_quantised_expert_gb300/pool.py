"""Slot pool: expert slots in one caller-owned device buffer.

The pool is a torch uint8 tensor on the device (PyTorch provides the memory);
each slot holds one expert (W1 | W3 | W2) in the device layout written by
bqe_pool_pack_slot, at a 256-byte-aligned offset.  Two small device tables
(slot byte offsets, slot formats) describe it to the kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _abi


class SlotPool:
    def __init__(self, d: _abi.bqe_layer_desc, slot_fmts, device="cuda"):
        self.d = d
        self.fmts = np.asarray(slot_fmts, dtype=np.int32)
        self.device = torch.device(device)
        sizes = [_abi.bqe_expert_bytes(d, int(f)) for f in self.fmts]
        if any(s == 0 for s in sizes):
            raise ValueError("bad layer shape or slot format")
        offs, o = [], 0
        for s in sizes:
            offs.append(o)
            o += (s + 255) // 256 * 256
        self.sizes = np.asarray(sizes, dtype=np.int64)
        self.offsets = np.asarray(offs, dtype=np.int64)
        self.nbytes = o
        self.buf = torch.empty(max(o, 256), dtype=torch.uint8, device=self.device)
        self.slot_off = torch.from_numpy(self.offsets.copy()).to(self.device)
        self.slot_fmt = torch.from_numpy(self.fmts.copy()).to(self.device)
        self._staging = None

    def __len__(self):
        return len(self.fmts)

    def slot_ptr(self, s: int) -> int:
        return self.buf.data_ptr() + int(self.offsets[s])

    def upload(self, s: int, canon, stream=None):
        """canon: canonical expert bytes (numpy uint8 on the host or a uint8 device tensor)."""
        n = int(self.sizes[s])
        if isinstance(canon, np.ndarray):
            if canon.size != n:
                raise ValueError("slot %d expects %d bytes, got %d" % (s, n, canon.size))
            if self._staging is None or self._staging.numel() < n:
                self._staging = torch.empty(n, dtype=torch.uint8, device=self.device)
            src = self._staging[:n]
            src.copy_(torch.from_numpy(np.ascontiguousarray(canon)))
        else:
            src = canon
            if src.numel() != n:
                raise ValueError("slot %d expects %d bytes, got %d" % (s, n, src.numel()))
        _abi.bqe_pool_pack_slot(self.d, int(self.fmts[s]), src, self.slot_ptr(s), stream)

    def cstruct(self) -> _abi.bqe_pool:
        return _abi.bqe_pool(self.buf.data_ptr(), self.nbytes, self.slot_off.data_ptr(), self.slot_fmt.data_ptr(),
                             len(self.fmts), 0)
