"""fp64 CPU oracle for the KDA forward pass (test infrastructure only)."""
