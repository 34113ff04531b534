"""CPU oracle for the BitLinear forward (test infrastructure only).

See ``oracle/bitlinear_oracle.py``. Only tests, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference legs use it; the product path
never imports it.
"""
from .bitlinear_oracle import *  # noqa: F401,F403
from .bitlinear_oracle import __all__  # noqa: F401
