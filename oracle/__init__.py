"""fp64 CPU oracle (test infrastructure only; never on the product path)."""
from .attention import attention_fwd, attention_rows, oracle_threads  # noqa: F401
from .backward import attention_bwd, attention_bwd_keys, attention_bwd_rows  # noqa: F401
