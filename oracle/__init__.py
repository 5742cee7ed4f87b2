"""Float64 CPU oracle (test infrastructure only; see ``oracle.attention``)."""
from . import attention  # noqa: F401
