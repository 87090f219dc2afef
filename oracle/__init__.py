"""Float64 CPU oracle of the TwoTower denoise step (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never links, imports or executes it,
and it imports nothing from the library.
"""
from .twotower import (UnmaskResult, commit_rule, context_rows, decode, denoise_attention,  # noqa: F401
                       denoise_attention_seq, kv_append, linear_schedule_mask, masked_nll,
                       masked_nll_seq, unmask, unmask_seq)
