"""KVarN K4V2 g128 KV-cache compression and paged decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libkvarn.so`` (hand-written CUDA kernels).
``calibration_free_kv_gb300.kvarn`` is the thin ctypes binding over it; importing
that module loads the library and raises if it has not been built.
"""

__all__ = ["kvarn", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
