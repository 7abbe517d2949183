"""fp64 CPU oracle for paged split-KV decode attention (test infrastructure only)."""
