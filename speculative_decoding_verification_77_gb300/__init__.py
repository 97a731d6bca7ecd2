"""GB300-native verification attention for long-context speculative decoding.

The compute path is the C-ABI library ``libspecverify.so`` (hand-written
sm_103a CUDA kernels) declared in ``include/specverify.h``; ``ops`` is its
thin PyTorch binding. ``workloads`` draws the seeded synthetic inputs.
Importing the package loads nothing; the first call into ``ops`` loads the
library and raises if it is missing.
"""

__all__ = ["ops", "workloads"]


def __getattr__(name):
    if name in ("ops", "workloads"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
