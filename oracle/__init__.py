"""fp64 CPU oracle for MLA decode (test infrastructure; see mla_oracle's header)."""
from .mla_oracle import *  # noqa: F401,F403
from . import mla_oracle  # noqa: F401
