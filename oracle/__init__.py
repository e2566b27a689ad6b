"""CPU fp64 oracle for the exact softmax attention forward and backward.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline and reference legs, never by the product path.
"""
from .oracle import Oracle, backward, build, compile_source, default_threads, forward, linear, probs  # noqa: F401
