"""Grouped differential attention on GB300 (sm_103a): Python binding (WIP)."""
import math


def lambda_init_schedule(layer: int) -> float:
    return 0.8 - 0.6 * math.exp(-0.3 * (layer - 1))
