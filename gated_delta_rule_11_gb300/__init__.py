"""GB300-native Kimi Delta Attention (KDA) operator.

The compute path is the C-ABI library ``libkda`` (hand-written CUDA for
sm_103a, sources in ``csrc/``); this package only marshals arguments to it.
"""
