"""fp64 CPU oracle of the eviction pass and the flat decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` import it; the library never does.
"""
from .kvevict_oracle import *  # noqa: F401,F403
from .kvevict_next import (capped_split, critical_positions_kappa, gqa_critical_kappa,  # noqa: F401
                           head_proj_norm, laprox_head_budgets, laprox_score, lava_cascade,
                           layer_top_from_held, reevict_rows, streaming_positions,
                           window_head_terms)
