"""CPU oracle of LSH-sampled decode attention (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import this
package. It shares no code with the CUDA library.
"""
from .magicpig_oracle import *  # noqa: F401,F403
from .magicpig_oracle import (HeadTables, center_of_keys, collision_probability,  # noqa: F401
                              decode_head, exact_attention, exact_tokens, expected_budget,
                              inclusion_probability, lsh_region, match_counts, near_ties,
                              projections, sampled_set, simhash_codes, snis_attention,
                              snis_logits, snis_sums, NEAR_TIE_REL, THRESHOLD)
