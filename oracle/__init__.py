"""CPU oracle for the convolution forward pass -- test infrastructure only.

Only ``tests/``, the package smoke check and the benchmark's CPU-baseline leg
use it.  See ``conv_oracle.c`` for the definition it follows.
"""
