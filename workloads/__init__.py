"""Seeded synthetic workloads shared by the tests, the benchmark and the oracle.

Holds sizes, counts and random draws only -- none of the method's arithmetic.
"""
from .configs import (ALL, BY_NAME, CTX_8K, CTX_32K, CTX_128K, TINY, VARLEN, Request, Workload,
                      request, small)
from .generate import Inputs, StepInputs, generate, generate_request

__all__ = ["ALL", "BY_NAME", "TINY", "CTX_8K", "CTX_32K", "CTX_128K", "VARLEN", "Workload",
           "small", "Inputs", "generate", "Request", "request", "StepInputs", "generate_request"]
