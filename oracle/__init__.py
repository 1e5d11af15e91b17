"""fp64 CPU oracle (test infrastructure only; never on the product path)."""
from . import mlp  # noqa: F401
