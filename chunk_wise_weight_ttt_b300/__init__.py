"""B300-native (sm_103a) In-Place TTT fast-weight MLP layer.

The layer's kernels live in ``libttt_mlp.so`` (C ABI: include/ttt_mlp.h);
``TTTMLP`` is a thin PyTorch-facing binding over it.
"""
from ._abi import TTTError, TTT_BF16, TTT_F32  # noqa: F401


def __getattr__(name):
    if name in ("TTTMLP", "TTTStack", "rmsnorm", "residual_add", "residual_rmsnorm", "workspace_bytes"):
        from . import layer
        return getattr(layer, name)
    raise AttributeError(name)
