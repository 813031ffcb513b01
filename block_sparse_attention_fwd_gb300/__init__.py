"""GB300-native BackLite attention: exact forward with per-tile LSE statistics,
tile selection (mask_from_stats) and a block-sparse backward.

The compute lives in ``libbl_attn.so`` (hand-written sm_103a CUDA behind the C
ABI in ``include/bl_attn.h``); this package only marshals arguments.  The
library is loaded on first use and a missing library raises.
"""
from . import _lib  # noqa: F401
from ._lib import (BLError, alloc_lists, attn_bwd, attn_fwd, bwd_check_status,  # noqa: F401
                   bwd_workspace_bytes, make_shape, mask_from_stats, tile_stats_elems, tiles)
from .api import BLAttention  # noqa: F401
