"""Test infrastructure: the plain CPU oracle for the deterministic attention backward.

This package is NOT part of the product. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it. It shares no code with the CUDA path:
the kernels never call it and it never calls them.

Modules
-------
attention : fp64 attention forward and backward, written out from the plain
            definition of softmax attention and its gradient.
dag       : the DASH task orders (ascending, descending Q-tile, shift, symmetric
            shift) and the critical path of the compute/reduce DAG, computed as a
            longest path over an explicit vertex/edge graph.
"""
