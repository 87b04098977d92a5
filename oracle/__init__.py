"""CPU oracle for FORGE's tile-fused weight-gradient + optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only the
tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may call it.  It shares no code with the CUDA path: it is a
plain, slow restatement of what the method computes, written from the
description in "FORGE: Fused On-Register Gradient Elimination for
Memory-Efficient LLM Training" (gist.science explainer, Technical Summary):

* weight gradient dW = dY^T X, accumulated here in float64 over the full matrix
  and rounded once to float32 (Technical Summary §2, "Core Mechanism":
  tile-wise gradient accumulation in FP32; "Exactness": the tiled update equals
  the full-gradient update up to the order of summation);
* the elementwise optimizer rule applied in float32 (§2 "In-Register
  Optimization", "Precision and Fidelity": the gradient is consumed in FP32);
* BF16 write-back by stochastic rounding keyed on (seed, step, element index)
  (§2 "Precision and Fidelity", dead-zone bullet);
* INT8 optimizer states in blocks of 64 (§2 "Precision and Fidelity", last
  bullet);
* dX = dY W from the pre-update weights (§5 "Limitations").

Modules:
  philox       Philox4x32-10 counter-based generator (Salmon et al., SC'11)
  rounding     bf16 round-to-nearest-even and stochastic rounding
  quant        block-64 absmax INT8 quantiser
  optimizers   the eight elementwise rules and their per-step scalars
  linear_step  the full step on one linear layer (and element-sampled variants)

Pins (see tests/test_oracle_*.py) tie each function to something outside itself:
closed forms, torch.optim run in float64, Triton's Philox run on the CPU
interpreter, brute-force exact sums on integer grids, statistical unbiasedness
of stochastic rounding, and hand-worked quantiser fixtures under tests/golden/.
"""

from . import philox, rounding, quant, optimizers, linear_step  # noqa: F401

__all__ = ["philox", "rounding", "quant", "optimizers", "linear_step"]
