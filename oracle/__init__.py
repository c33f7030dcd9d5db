"""fp64 CPU oracle (test infrastructure only; see ``kl_oracle``)."""
from .kl_oracle import *  # noqa: F401,F403
from .kl_oracle import bf16_bits_to_f64, forward, backward  # noqa: F401
