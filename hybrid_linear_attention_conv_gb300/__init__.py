"""Gated DeltaNet mixer for GB300 (sm_103a): decode, tree verify, commit and
chunked prefill as hand-written CUDA kernels behind a C ABI (``include/gdn.h``).

``inputs`` holds the seeded synthetic input generator; ``gdn`` is the thin
Python binding over the shared library (loaded on first use, and an error if it
is missing -- there is no CPU fallback).
"""
