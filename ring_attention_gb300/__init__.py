"""Blockwise exact attention for GB300 (sm_103a): a C-ABI CUDA library and its binding.

``ring_attention_gb300.bpa`` loads ``libbpa.so`` (built by
``ring_attention_gb300.build``) and exposes its entry points;
``ring_attention_gb300.inputs`` draws the seeded synthetic workloads.
Importing the package loads nothing.
"""
