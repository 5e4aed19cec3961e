"""Float64 CPU oracle for the M2RNN scans (test infrastructure only).

Only the test-suite, the package entry module's smoke check and the benchmark's
CPU-baseline leg import this package.  See ``m2rnn_oracle`` for the equations
and their sources.
"""
from .m2rnn_oracle import (backward, forward, gate, gate_backward, loss, output_norm,  # noqa: F401
                           output_norm_backward)
