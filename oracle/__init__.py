"""CPU oracle for the RidgeFill fill and fit (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The library never imports it, and it imports nothing from the
library.
"""
from .ridgefill import (  # noqa: F401
    ridge_fit,
    fit_sums,
    ridge_solve_from_sums,
    rms_norm,
    rope_rotate_half,
    late_layer_kv,
    map_apply,
    fill_attention,
    kv_rescale,
    gdn_projections,
    gdn_recurrence,
    gdn_state,
    speedup_ceiling,
    filled_weight_share,
    filled_share,
    gdn_rho,
    terminal_correction,
    layer_inputs,
    quantize_map,
    dequantize_map,
    Q8_GROUP,
)
