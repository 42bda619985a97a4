"""Block-quantised MoE expert layer for GB300 (sm_103a).

The compute lives in libbqe.so (CUDA, include/bqe.h).  This package is its
thin Python face: `_abi` binds the C entry points under their own names,
`pool` lays expert slots out in a caller-owned device buffer (PyTorch tensors
serve as device memory).  Importing `bit_quantised_expert_gb300._abi` fails
loudly when the library is not built.
"""
__all__ = ["build", "abi", "pool"]


def build(force: bool = False):
    from . import buildlib as _b
    return _b.build(force=force)
