"""GB300-native (sm_103a) forward of a mixture-of-experts FFN layer with
groupwise-affine 4-bit expert weights and GPU-resident routing.

The kernels live in libmoe_w4.so (csrc/, C ABI in include/moe_w4.h); this
package only binds them (``_lib``) and wraps one layer (``layer.MoELayerW4``).
"""
from . import _lib  # noqa: F401
from ._lib import MoeError, load  # noqa: F401

__all__ = ["MoeError", "load", "MoELayerW4"]


def __getattr__(name):
    if name == "MoELayerW4":
        from .layer import MoELayerW4
        return MoELayerW4
    raise AttributeError(name)
