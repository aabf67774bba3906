"""TQ1_0 ternary mat-vec for GB300 (sm_103a): Python binding of libtq1.

Importing the package loads nothing; the CUDA library is loaded on first use
of a binding function (see ``_lib``).
"""
