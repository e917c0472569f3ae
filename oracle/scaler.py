"""ORACLE -- test infrastructure.  The dynamic loss-scale policy in plain float32 arithmetic.

After each reduction: on overflow the scale is multiplied by the back-off factor (kept >= min_scale) and the
count of clean steps restarts; after growth_interval consecutive clean steps it is multiplied by the growth
factor (kept <= max_scale).  The pages only name loss scaling as state to keep and align; this is the
growth/back-off rule of common mixed-precision scalers, with the range clamp the sweep workload asks for.
"""
import numpy as np


def update(scale: float, good: int, found: bool, growth: float, backoff: float, interval: int,
           min_scale: float, max_scale: float):
    s = np.float32(scale)
    if found:
        return float(max(np.float32(s * np.float32(backoff)), np.float32(min_scale))), 0
    if good + 1 >= interval:
        return float(min(np.float32(s * np.float32(growth)), np.float32(max_scale))), 0
    return float(s), good + 1
