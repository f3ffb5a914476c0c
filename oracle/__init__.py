"""Float64 CPU oracle for MLA verify attention.

Test infrastructure: only the tests, the package's smoke check and the
benchmark's CPU-baseline leg use it.  The GPU library never imports it.
"""

from .mla_oracle import (  # noqa: F401
    BRANCH_ABSORBED, BRANCH_MATERIALISED, MODE_ABSORBED, MODE_AUTO, MODE_MATERIALISED,
    absorbed, brute_force, default_scale, gather_paged, materialised,
    max_absorbed_queries, max_absorbed_queries_batch, select_branch, sparse_absorbed,
)
from .draft_cap import accepted, select_draft_cap  # noqa: F401
from . import indexer_pool, rollback_state  # noqa: F401
