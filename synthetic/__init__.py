"""Seeded synthetic inputs (no attention arithmetic); see txl_inputs."""
from .txl_inputs import *  # noqa: F401,F403
