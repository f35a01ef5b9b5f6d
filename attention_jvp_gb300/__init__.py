"""GB300-native forward-mode JVP through softmax attention.

The compute path is a C-ABI shared library (``csrc/`` -> ``libattnjvp.so``)
of hand-written sm_103a kernels; ``binding`` marshals torch tensors into it.
"""
