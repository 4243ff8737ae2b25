"""GB300-native (sm_103a) batch-invariant attention core of a MiniMax-H3 DiT block.

``h3attn`` is the Python binding of the C-ABI library ``libh3attn.so``;
``workloads`` builds seeded synthetic inputs.
"""
