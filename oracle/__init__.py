"""fp64 CPU oracle for the AKV cache operations — TEST INFRASTRUCTURE ONLY.

A plain, slow restatement of what the pages of "Cache Engineering for
Agents" (arXiv 2610.28577) define, used to check the CUDA library:

* ``replay``            the cache-operation sequence (append / drop / repos)
                        run from an empty cache, operate-after, drop before
                        repos at one boundary (paper section 3.3-3.4, Figure 6);
* ``replay_attention``  single-layer attention of every token over the active
                        cache at its append time (the sequential definition);
* ``segment_batch_attention`` the same result by the segment-batch rule of
                        section 4.2 / Appendix A.1.1, derived from the op log
                        by formula (used to cross-check the replay);
* ``repos_rotate``      K_q = R(q - p) K_p, V unchanged (section 3.3);
* ``compact``           active logical indices and positions at a boundary;
* ``decode_attention``  one query per request over a page-size-1 pool;
* ``model_replay``      a multi-layer decoder replayed message by message.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
may import this package.  The CUDA library never calls it, and it shares no
code with the library.  Every function computes in float64.
"""
from .core import (  # noqa: F401
    OpLogError,
    widen,
    rope,
    validate,
    replay,
    replay_attention,
    visible_counts,
    compact,
    repos_rotate,
    decode_attention,
)
from .segment_batch import segment_tables, segment_batch_attention  # noqa: F401
from .model import model_replay, rmsnorm  # noqa: F401
