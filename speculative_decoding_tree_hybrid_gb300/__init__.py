"""GB300-native Hybrid Tree Attention (tree-verification attention for
speculative decoding), shipped as the C-ABI library ``libhta`` plus a thin
ctypes binding. The binding is loaded on first use so that the seeded
workload generators can be imported on machines without a GPU.
"""
