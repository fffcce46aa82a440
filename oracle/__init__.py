"""fp64 CPU oracle (test infrastructure; never used by the product path)."""
