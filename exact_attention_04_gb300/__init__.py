"""Exact attention (FlashAttention-style) for one NVIDIA GB300 (sm_103a).

``exact_attention_04_gb300.fa`` is the thin binding over the C-ABI library
``libfa.so`` (built from ``csrc/`` by ``exact_attention_04_gb300.build``);
``exact_attention_04_gb300.workloads`` draws the seeded synthetic inputs.
Importing the package loads nothing: the library is opened on first use and
the call fails loudly if it is missing.
"""
__all__ = ["fa", "workloads", "build"]
