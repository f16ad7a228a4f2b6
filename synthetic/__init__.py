"""Seeded synthetic inputs for the late-layer cache fill and the ridge fit.

This package only draws random numbers and lays them out in the tensor
layouts the library and the oracle both read.  It computes nothing that the
fill or the fit computes.
"""
from .workloads import (  # noqa: F401
    FillShape,
    GdnShape,
    WORKLOADS,
    normal,
    channel_scales,
    fill_inputs,
    tail_inputs,
    exact_rows,
    true_inputs,
    gdn_inputs,
    calibration,
    calibration_device,
    to_f64,
)
