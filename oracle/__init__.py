"""Plain fp64 CPU oracle for SnapKV observation-window KV selection.

Test infrastructure only: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never does.
"""

from .snapkv_oracle import (  # noqa: F401
    OracleArgumentError,
    causal_probabilities,
    check_head_args,
    pool_scores,
    prefix_votes,
    select_from_pooled,
    snapkv_head,
    snapkv_packed,
    top_prefix,
    window_logits,
    window_row_exp_sums,
)
from .gqa_oracle import snapkv_group, snapkv_packed_gqa  # noqa: F401,E402
from .decode_oracle import (  # noqa: F401,E402
    cache_lengths,
    decode_attention,
    decode_packed,
    decompose,
    full_probabilities,
)
from .jacap_oracle import (  # noqa: F401,E402
    capacity_matrix,
    jacap_head,
    leverage,
    weights,
    window_statistics,
)
from .reverse_oracle import reverse_attention, reverse_packed  # noqa: F401,E402
