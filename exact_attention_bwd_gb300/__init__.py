"""Exact softmax attention (forward and backward) for one GB300, sm_103a.

The compute path is the CUDA library ``libfa_gb300.so`` behind the C ABI in
``include/fa.h``; :mod:`exact_attention_bwd_gb300.binding` marshals arguments
to it.  The library is loaded on first use and its absence is an error: there
is no CPU fallback.
"""
