"""Float64 CPU oracle for the M2RNN scans (test infrastructure only).

Only the test-suite, the package entry module's smoke check and the benchmark's
CPU-baseline leg import this package.  See ``m2rnn_oracle`` for the equations
and their sources.
"""
from .m2rnn_oracle import backward, forward, loss  # noqa: F401
