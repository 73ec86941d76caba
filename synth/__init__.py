"""Seeded synthetic input generators shared by the tests, the bench and the oracle's
callers.  Holds no attention arithmetic."""
from .inputs import *  # noqa: F401,F403
from .inputs import WORKLOADS, HEAD_DIM  # noqa: F401
