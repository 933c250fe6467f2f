"""CPU oracle for the prefix-tree training hot path — TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 NumPy restatement of what the path computes, written from
the tree-training pages:

* ``oracle.tree``      — DFS serialisation of the rollout tree, per-token
  ancestor sets, leaf-fraction weights, interval lists ("Tree Training",
  Abstract: DFS serialization, per-token weights).
* ``oracle.attention`` — causal attention restricted to each token's
  root-to-token path, forward and backward, by linearising every branch
  ("Tree Training", Abstract: log-probs match independent per-branch
  calculation; AReaL-DTA, Key Contributions 1: gradients from all descendant
  leaves accumulate into the shared prefix).
* ``oracle.logprob``   — per-branch log-softmax loss averaged over branches and
  the equivalent per-token weighted loss ("Tree Training", Abstract).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. It shares no code with the CUDA library
(``prefix_tree_gb300``) and never imports it; its only common dependency is
the input generator module ``synth``, which holds no arithmetic of the method.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against hand-derived fixtures, closed forms, brute force or library routines
(PyTorch fp64 SDPA / autograd / log_softmax); none is "parity unpinned".
"""
