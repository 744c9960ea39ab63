"""CPU oracle of the MoE FFN layer forward (test infrastructure only: imported by
the tests, the smoke check and the benchmark's CPU-baseline leg, never by the
product path)."""
