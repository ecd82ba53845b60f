"""Exact IO-aware attention for GB300 (sm_103a): forward with online softmax + LSE,
recomputing backward, behind the C ABI of ``libfa.so``."""
