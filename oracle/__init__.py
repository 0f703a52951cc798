"""Float64 CPU oracle (test infrastructure; see attention_oracle.py)."""
from .attention_oracle import *  # noqa: F401,F403
from .attention_oracle import (allowed, alibi_slope, backward, classify_tiles,  # noqa: F401
                               document_ids, forward, probabilities, allowed_pairs)
