"""Oracle (TEST INFRASTRUCTURE ONLY): a plain fp64 CPU statement of the indexer -> Top-K ->
sparse-attention chain.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
may import it; the product path never does."""
from .dsa_oracle import *  # noqa: F401,F403
from . import parity  # noqa: F401
