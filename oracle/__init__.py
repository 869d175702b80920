"""fp64 CPU oracle for HSTU jagged causal attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import anything from
this package.  The product path (``hstu_jagged_attention_gb300``) never
imports it, and the two share no code: no kernels, headers, helpers or
constant tables.  Only the seeded input generator
(``hstu_jagged_attention_gb300.workloads``) feeds both.

Contents
--------
``reference``  -- ctypes wrapper of ``hstu_oracle.c``: the jagged formula
                  summed row by row in fp64 (all rows, or sampled rows).
``dense``      -- the padded-dense brute force: the post's PyTorch definition
                  (score matmul, scale, SiLU, multiplicative tril mask and 1/n,
                  matmul with V) evaluated with numpy float64 on (b, heads, s, s)
                  tensors.  Used to pin ``reference`` on tiny inputs.
``worklist``   -- plain Python enumeration of the (sequence, head, q-tile)
                  work items in longest-first order.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
something other than itself (closed forms, limits, library routines, brute
force, invariants).
"""
