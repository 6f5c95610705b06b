"""fp64 CPU oracle for the decode-time skinny linears (test infrastructure only)."""
