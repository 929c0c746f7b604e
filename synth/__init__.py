"""Seeded synthetic inputs for the CSA hot path.

This package holds no step of the method's arithmetic: it only draws the tensors
(Gaussian activations, compressed caches, gates, sinks) that both the CPU oracle and
the CUDA library read.  See :mod:`synth.gen`.
"""
from .gen import CONFIGS, CsaConfig, make_inputs, normal, uniform01  # noqa: F401
