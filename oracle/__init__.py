"""CPU oracle of the decode-step attention block — test infrastructure, not product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package. It never imports the CUDA package and the
CUDA package never imports it.
"""
from . import brute, decode_ref  # noqa: F401
