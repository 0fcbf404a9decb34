"""Seeded synthetic input generation shared by the oracle and the GPU path."""
