"""fp64 CPU oracle (test infrastructure only; see ``oracle.oracle``)."""
from .oracle import bf16_to_f64, sparse_mla_fwd, token_forward, valid_slots  # noqa: F401
