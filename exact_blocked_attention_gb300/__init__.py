"""Exact blocked attention over a KV cache for GB300 (sm_103a).

The compute path lives in the C-ABI library ``libblkattn.so`` built from
``csrc/``; :mod:`exact_blocked_attention_gb300.blkattn` is its thin Python
binding (argument marshalling only).  :mod:`.workloads` draws seeded synthetic
inputs.  Importing the package loads nothing; the library is loaded on the
first call and a missing build is an error, never a fallback.
"""
