"""Float64 CPU oracle for the tree-verify step (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package; the product path never does.
"""
