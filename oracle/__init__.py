"""fp64 CPU oracle for the H2O decode / prefill path.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product path.
"""
