"""Seeded input generators shared by the oracle tests and the CUDA path (no method arithmetic)."""
