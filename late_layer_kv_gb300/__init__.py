"""RidgeFill late-layer cache fill and ridge fit for GB300 (sm_103a).

The compute lives in the C-ABI library ``lib/libridgefill.so`` (hand-written
CUDA kernels, see ``include/ridgefill.h``); :mod:`.ridgefill` is a thin ctypes
binding with the same names.
"""
from .ridgefill import (  # noqa: F401
    FitSums,
    RidgeFillError,
    compute_share,
    debug_library,
    device_error,
    load,
    library_path,
    ridgefill_fill,
    ridgefill_fill_gdn,
    ridgefill_fit_accumulate,
    ridgefill_fit_solve,
    ridgefill_quantize_maps,
    ridgefill_rescale,
    Q8_GROUP,
    RF_RESCALE_KEYS,
    RF_RESCALE_VALUES,
    ridgefill_workspace_size,
    wait_selftest,
)
