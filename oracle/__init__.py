"""fp64 CPU oracle of the ReLU RNN forward recurrence -- test infrastructure
only (tests, the smoke check and the benchmark's CPU-baseline leg)."""
from .oracle import Oracle, compile_oracle, default  # noqa: F401
