"""Helpers shared by the tests (re-exported from the workload module, which
holds the glue that replays a workload's add/remove program on a state)."""
from pkv_workloads import apply_ops, group_tuples, schedule_arrays  # noqa: F401
