"""CPU oracle for the C2KV hot path: test infrastructure, never product code."""
