"""CPU oracle for the fused IQL + HER offline-RL train step.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the train step computes, in numpy with fp64 arithmetic
(fp32 only where the method itself fixes fp32: the HER goal-distance test).
Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import it.  The CUDA library never calls it and shares no code with it;
the two meet only through the seeded inputs of the `synth` package.

Sources (web pages describing the method):
  * "GPU IQL + HER Porting Plan": IQL value network, expectile loss,
    advantage-weighted policy, HER relabel, donor strategies, Adam launch.
  * "DQN Backward-Path NaN Audit": Adam semantics (non-finite guard, clip
    formula, bias correction with t >= 1, norm as a raw sum of squares).
  * "Gradient Stability -- Multi-Task Gradient Isolation + Full Spectral
    Norm": budgeted per-source clipping (0.70/0.15/0.10/0.05) and its order.

Every function states the passage it follows.  Pins for every function live
in tests/test_oracle_*.py.
"""
from . import her, iql, optim, precision, rng, step  # noqa: F401
