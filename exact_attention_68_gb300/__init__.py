"""GB300-native fused exact attention forward (sm_103a).

The compute path is the C-ABI library ``libattn_sm103.so`` built from
``csrc/``; this package only marshals arguments to it (see ``binding``).
"""
