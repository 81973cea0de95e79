"""GB300-native UniPrefill token selection (libupf) and its Python binding.

* ``_binding``: ctypes binding of the C ABI in ``include/upf.h`` (same names).
* ``selector``: torch-tensor front end (``TokenSelector.select_tokens``).
* ``tp``: heads sharded over tensor-parallel ranks, one score all-reduce.
* ``workload``: seeded synthetic inputs (no method arithmetic).
* ``build``: compiles ``libupf.so`` in-tree for sm_103a.

Importing the package loads nothing; the library is loaded on first use and a
missing library raises.
"""
import importlib

__all__ = ["workload", "build", "_binding", "selector", "tp", "TokenSelector"]


def __getattr__(name):
    if name in ("workload", "build", "_binding", "selector", "tp"):
        return importlib.import_module(f".{name}", __name__)
    if name == "TokenSelector":
        return importlib.import_module(".selector", __name__).TokenSelector
    raise AttributeError(name)
