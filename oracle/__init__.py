"""CPU oracle (test infrastructure only; the library never imports it)."""
from .akv_oracle import (OracleCache, OracleError, inv_freq, rope, rope_inverse,
                         reposition_key, rne_bf16, to_pool)

__all__ = ["OracleCache", "OracleError", "inv_freq", "rope", "rope_inverse",
           "reposition_key", "rne_bf16", "to_pool"]
