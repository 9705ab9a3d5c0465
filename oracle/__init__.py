"""CPU oracle for the chunkwise Gated DeltaNet forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or run anything in this package.  The CUDA
library never does, and nothing here imports the CUDA library: the two share no
code, headers, tables or helpers.  Only the seeded input generator
(``workloads.py``) serves both sides.

Contents (fp64 throughout):

* ``recurrence``  -- the definition: the per-token Gated DeltaNet recurrence
  (qiita Nyysyyan, "Gated-DeltaNet" section, the update S_i = a_i S_{i-1}
  (I - b_i k_i k_i^T) + b_i v_i k_i^T with read h_i = S_i q_i), plus the gate ->
  predict -> delta -> write statement of the same layer from kkkzoz
  "linear-attention", "Gated DeltaNet" and "Workflow" sections.
* ``derivations`` -- the page's own closed forms and identities used to pin the
  recurrence: linear attention and Mamba2 matrix forms, the WY identity, the U/G
  identity, the unrolled state, the full-sequence matrix form and the chunk
  computation, and the chunk form's backward (pinned to ``backward``).
* ``backward``    -- the reverse-mode derivative of the per-token recurrence
  (gradients of q, k, v, log alpha, beta and S0 for given output and final-state
  gradients); the pages derive none, so it is pinned to finite differences and to
  autograd of a separately written forward.
* ``native``      -- the same recurrence in plain C with OpenMP over
  (sequence, head), for sizes numpy is too slow for; built by ``oracle/build.py``.

Pinning status: every function here is pinned by ``tests/test_oracle_pins.py``
against a closed form, an identity, an invariant or brute force; none is
"parity unpinned".
"""
