"""Scalar CPU oracle of the Q8_0 decode path (test infrastructure only)."""
