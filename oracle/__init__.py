"""Float64 CPU oracle of the Kamera reuse operator (test infrastructure only).

Imported by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and reference legs;
the library never imports it.
"""
from .kamera_oracle import *  # noqa: F401,F403
from . import kamera_oracle  # noqa: F401
