"""GB300-native causal log-linear Mamba-2 attention.

The compute lives in ``liblla.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/lla.h``); :mod:`log_linear_attention_gb300.binding` marshals
torch tensors into those calls. Importing this package loads nothing: the
library is loaded on first use and a missing library is an error, never a
fallback.
"""
__all__ = ["binding", "inputs"]
