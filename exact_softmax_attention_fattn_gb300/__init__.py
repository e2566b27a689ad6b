"""Exact softmax attention forward for GB300 (sm_103a).

The compute path is one hand-written CUDA kernel behind the C ABI declared in
include/fattn.h (libfattn.so); `forward` is the thin Python binding over it.
The binding is imported on first use so that the input generator can be used
without the CUDA library.
"""
_BINDING_NAMES = (
    "FattnError",
    "forward",
    "forward_into",
    "last_error",
    "library_path",
    "load_library",
    "status_string",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
