"""CPU oracle of the EAGLE-2 draft-tree verification step.

TEST INFRASTRUCTURE ONLY: plain float64 / integer restatement of the method,
used to check the CUDA path.  Only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) may import
it; the library never does, and it never imports the library.
"""
from .eagle_tree_oracle import *  # noqa: F401,F403
from .eagle_tree_oracle import (TreeCfg, Tree, AcceptResult, GREEDY, STOCH_POINT, STOCH_DRAFTQ,  # noqa: F401
                                FRAC_BITS, KEY_MIN)
from .kv_commit_oracle import kv_commit  # noqa: F401
from .static_tree_oracle import static_tree, static_tree_sampled, static_depths  # noqa: F401
from .lm_head_oracle import lm_head_logits, lm_head_error_bound  # noqa: F401
