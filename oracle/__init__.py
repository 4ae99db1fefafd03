"""CPU oracle of the DFlash draft-and-verify cycle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  See ``dflash_oracle`` for the method
and the readings it takes.
"""
from .dflash_oracle import *  # noqa: F401,F403
from .dflash_oracle import (Weights, Model, feature_layers, spec_generate, greedy_generate,  # noqa: F401
                            target_forward, draft_blocks, fuse_features, inject_kv, accept_prefix)
