"""fp64 CPU oracle of the tensor-parallel sharded linear block.

TEST INFRASTRUCTURE: imported only by the tests, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference arm; never by the library.
"""
from .tp_oracle import *  # noqa: F401,F403
from .tp_oracle import (COLUMN, ROW, VOCAB, REPLICATED, NO_COMM, ALL_REDUCE,  # noqa: F401
                        ALL_GATHER, REDUCE_SCATTER, WEIGHTS, PlanError, RankShard, RingLog)
