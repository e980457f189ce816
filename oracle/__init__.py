"""CPU oracle (test infrastructure only; never on the product path)."""
from .ttt_ref import OracleConfig, prefill, full_forward_losses  # noqa: F401
