"""TokenGate gated prefill on B300 (sm_103a): the C library libtokengate.so
and its Python binding.  See include/tokengate.h for the C ABI."""
from .tokengate import *  # noqa: F401,F403
from .tokengate import __all__  # noqa: F401
