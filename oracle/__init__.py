"""fp64 CPU oracle for exact attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The library's compute path never calls it.
"""
from .attention import attention_head, attention, attention_probs  # noqa: F401
from .attention_bwd import (attention_bwd_head, attention_bwd, attention_bwd_query_rows,  # noqa: F401
                            attention_bwd_key_rows)
from .direct_p import direct_p_head, direct_p_probs  # noqa: F401
