"""CPU oracle for the packed BitLinear product (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path never does.
"""
