"""Slot pool: expert slots in one caller-owned device buffer.

PyTorch provides the memory (a uint8 tensor on the device); the library lays
the pool out (bqe_pool_bytes / bqe_pool_init: the slot-offset and slot-format
tables at the front, then every slot 256-byte aligned) and writes each expert
into its slot in the device layout (bqe_pool_upload).  Nothing here computes
offsets or sizes.
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
        nbytes = _abi.bqe_pool_bytes(d, self.fmts)
        if nbytes == 0:
            raise ValueError("bad layer shape or slot format")
        self.mem = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.pool = _abi.bqe_pool_init(d, self.fmts, self.mem, nbytes)
        self.sizes = np.array([_abi.bqe_expert_bytes(d, int(f)) for f in self.fmts], dtype=np.int64)
        self._staging = None

    def __len__(self):
        return len(self.fmts)

    def slot_ptr(self, s: int) -> int:
        """Device address of slot s, from the pool's own offset table."""
        at = int(self.pool.slot_off) - self.mem.data_ptr()
        off = self.mem[at:at + 8 * len(self.fmts)].view(torch.int64)[int(s)].item()
        return int(self.pool.base) + int(off)

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
        _abi.bqe_pool_upload(self.pool, self.d, int(s), src, stream)

    def cstruct(self) -> _abi.bqe_pool:
        return self.pool
