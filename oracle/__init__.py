"""Oracle of the routed MoE expert layer: plain, slow, float64, CPU.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package. The CUDA
path never imports it and shares no code, header, table or helper with it.

Modules:
  moe_oracle   the definition, forward and backward (numpy float64)
  bruteforce   a scalar-loop twin for tiny shapes (pins moe_oracle)
  sampled      single outputs of a large layer, evaluated from the definition
  calibrate_zipf  script: the router-bias temperature of the skewed workloads

Parity status: every function is pinned by the tests in
``tests/test_oracle_*.py`` (brute force, closed forms, the dense-MLP special
case, permutation and adjoint invariants, finite differences). The absolute
output values of the large workloads have no printed worked example on the
pages to compare against; they rest on the definition and these pins.
"""
