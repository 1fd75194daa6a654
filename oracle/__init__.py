"""fp64 CPU oracle (test infrastructure only; see ``mnb_oracle``)."""
from .mnb_oracle import *  # noqa: F401,F403
