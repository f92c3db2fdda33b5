"""MoE layer hot path for GB300 (sm_103a): route -> EPLB map -> dispatch ->
grouped FP8 FFN (tcgen05) -> combine, behind the C ABI of libmoe.so.

``api`` holds the Python names of the C entry points.  Importing the package does
not load the CUDA library; the first ``api`` call does, and raises if it is missing.
"""
from . import api, configs, inputs  # noqa: F401

__all__ = ["api", "configs", "inputs"]
