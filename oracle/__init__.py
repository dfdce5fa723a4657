"""CPU oracle of the sparse-decode path (test infrastructure; see hashattn_oracle)."""
from . import hashattn_oracle  # noqa: F401
