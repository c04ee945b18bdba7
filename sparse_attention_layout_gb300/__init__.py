"""Block-sparse SDD / DSD / DDS matmul, block-sparse row softmax and
block-sparse attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libbsp.so`` (hand-written CUDA);
``sparse_attention_layout_gb300.bsp`` is its thin Python binding and
``sparse_attention_layout_gb300.blocksparse`` the differentiable matmul /
softmax objects built on it.  The
library is loaded on first use and its absence is an error: there is no CPU
fallback.
"""

import importlib

__all__ = ["bsp", "blocksparse", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
