"""CPU oracle (test infrastructure only; see kk_oracle's header)."""
from . import kk_oracle  # noqa: F401
