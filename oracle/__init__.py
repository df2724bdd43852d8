"""CPU oracle of the fused MoE router (test infrastructure only: used by the
tests, the smoke check and the benchmark's CPU-baseline leg, never by the
product path)."""
