"""fp64 CPU oracle (test infrastructure; never on the product path)."""
