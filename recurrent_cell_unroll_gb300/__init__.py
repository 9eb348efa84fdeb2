"""GB300-native time-unrolled recurrent cells (LSTM, GRU, LSTMP, RSSM prior).

The compute lives in ``librcu.so`` (CUDA kernels for sm_103a behind the C ABI
in ``include/rcu.h``); ``binding`` is its thin ctypes binding.  Importing the
package does not load the library: the first binding call does, and fails
loudly if the library has not been built.
"""

__all__ = ["binding", "workloads", "build"]


def build(verbose: bool = False) -> str:
    from . import _build
    return _build.build(verbose=verbose)
