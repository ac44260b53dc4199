"""Seeded synthetic KV-cache inputs shared by the tests, the bench and the
oracle checks.  Holds no codec arithmetic."""
from . import workloads, synth  # noqa: F401
