"""CPU oracle (test infrastructure only; see rkv_oracle's header)."""
from .rkv_oracle import *  # noqa: F401,F403
from .rkv_oracle import __all__  # noqa: F401
