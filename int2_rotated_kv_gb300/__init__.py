"""GB300-native OSCAR mixed-precision INT2 KV cache: rotate+quantise+pack and
split-K paged decode attention, as a C-ABI library (include/oscar.h) with a thin
ctypes binding (``int2_rotated_kv_gb300.oscar``).

Importing the package does not load the library; ``from int2_rotated_kv_gb300
import oscar`` does, and fails loudly when it has not been built.
"""


def __getattr__(name):
    if name == "oscar":
        from . import _lib
        _lib.lib()
        return _lib
    raise AttributeError(name)
