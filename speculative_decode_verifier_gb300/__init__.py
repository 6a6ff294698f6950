"""GB300-native target-verifier step of lossless p/q speculative decoding.

The compute lives in ``libq2v.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/q2v.h``); ``q2v`` is the thin ctypes binding with the same
entry-point names.  ``synth`` draws the seeded synthetic inputs.  Nothing here falls
back to the CPU: a missing library is an error.
"""

__all__ = ["q2v", "synth"]


def __getattr__(name):
    if name in ("q2v", "synth"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
