"""Seeded synthetic workloads for the MSA forward pass.

This package only draws random inputs; it holds none of the method's
arithmetic, so the oracle and the CUDA path can both consume its output
without sharing any computation.  See ``configs.py`` for the shapes and
``generate.py`` for the recipe.
"""
from .configs import CONFIGS, Workload, get
from .generate import Inputs, PrologueInputs, generate, prologue_inputs

__all__ = ["CONFIGS", "Workload", "get", "Inputs", "PrologueInputs", "generate", "prologue_inputs"]
