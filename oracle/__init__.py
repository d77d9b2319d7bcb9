"""fp64 CPU oracle (test infrastructure only; see ``mla_oracle``).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""
from .mla_oracle import (  # noqa: F401
    D_LATENT, D_ROPE, D_QK, D_V, to_f64, gather_history, gather_history_fast,
    shard_bounds, segment_attention, decode_partials, lse_combine, v_up,
    decode_reference)
