"""GB300-native dynamic block-sparse attention (BSA) forward.

``plan`` maps a logical u8 block mask onto 128-row physical tiles (retain,
combine or subdivide) and emits a per-(head, q-tile) CSR list of K/V tiles, a
longest-row-first schedule and an optional GQA union table; ``forward`` runs a
persistent tcgen05/TMA kernel over exactly those tiles.  Both run in libbsa.so
(include/bsa.h); this package is its ctypes binding plus the seeded workload
generators.
"""
from ._lib import (  # noqa: F401
    BsaError, Layout, Plan, PLAN_NO_UNION, PLAN_Q64, PLAN_REMAP, STAGE_ALL, STAGE_BOUNDED, STAGE_EXACT, STAGE_KNORM, STAGE_PREPARE,
    STAGE_ROWBOUND, attention, attention_static, attention_static_status, forward, library, plan, plan_affine,
    plan_check, plan_layout, plan_workspace_bytes, select_flags, sync_status, watchdog_selftest,
)

__all__ = ["BsaError", "Layout", "Plan", "PLAN_NO_UNION", "PLAN_Q64", "PLAN_REMAP", "STAGE_ALL", "STAGE_BOUNDED",
           "STAGE_EXACT", "STAGE_KNORM", "STAGE_PREPARE", "STAGE_ROWBOUND", "attention", "attention_static", "attention_static_status", "forward", "library",
           "plan", "plan_affine", "plan_check", "plan_layout", "plan_workspace_bytes", "select_flags", "sync_status",
           "watchdog_selftest"]
