"""Exact attention for GB300 (sm_103a): tiled online-softmax forward and
recompute-based backward behind the C ABI of libfa.so.

``exact_attention_21_gb300.fa`` binds the library; ``inputs`` draws the seeded
synthetic workloads; ``build`` compiles the library in-tree.
"""
