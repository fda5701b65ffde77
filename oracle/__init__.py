"""fp64 CPU oracle of the parallel transformer block (test infrastructure only)."""
