"""GB300 (sm_103a) M2RNN forward/backward scans behind a C ABI (libm2rnn.so).

``binding`` holds the ctypes wrappers of the C ABI and the torch helpers;
``inputs`` holds the seeded synthetic input generator.  The library is loaded
on first use and its absence is an error: there is no fallback path.
"""
import importlib

from . import inputs  # noqa: F401

__all__ = ["inputs", "binding"]


def __getattr__(name):
    if name == "binding":
        return importlib.import_module(".binding", __name__)
    raise AttributeError(name)
