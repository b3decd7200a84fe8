"""CPU oracle for the ternary projection linears -- test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg,
never by the library.  Functions without an independent pin are marked
"parity unpinned" in their docstring; at present every function is pinned by
tests/test_oracle.py.
"""
