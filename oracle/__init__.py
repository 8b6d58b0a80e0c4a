"""fp64 CPU oracle for prefix-tree attention -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The library and its Python binding never do.
"""
