"""fp64 CPU oracle (test infrastructure only; never on the product path)."""
from .cf_oracle import *  # noqa: F401,F403
from .cf_oracle import __all__  # noqa: F401
