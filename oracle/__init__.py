"""fp64 CPU oracle (test infrastructure only; never on the product path)."""
from .attention import attention_fwd, attention_rows, oracle_threads  # noqa: F401
