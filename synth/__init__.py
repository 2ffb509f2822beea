"""Seeded synthetic inputs for the routed-MoE slot-pool layer.

This package only *draws* inputs: weights, router biases, hidden states and the
initial slot fill.  It holds none of the layer's arithmetic (no gating, no
SwiGLU, no scores), so the CPU oracle and the CUDA path can both consume what
it makes without sharing any of the method.  Shapes follow the five workload
shapes used throughout the project (see ``synth.configs``).
"""
from .configs import WORKLOADS, Workload, get_workload  # noqa: F401
from . import gen  # noqa: F401
