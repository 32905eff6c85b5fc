"""fp64 CPU oracle for attention forward, first backward and BoB.

Test infrastructure only: see ``oracle.attention``.
"""
from .attention import *  # noqa: F401,F403
from .attention import bob_sampled_rows  # noqa: F401
