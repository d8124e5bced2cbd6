"""Seeded synthetic workloads shared by the tests, the benchmark and the oracle."""
from .configs import ALL, BY_NAME, BUDGETED, HER_HEAVY, PROD, TINY, TWIN, Workload  # noqa: F401
from .gen import make_aux, make_params, make_q, make_replay, scaled  # noqa: F401
