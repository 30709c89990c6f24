"""Float64 CPU oracle for the LoongTrain 2D-Attention ring step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (no kernels, headers, helpers or constant tables).

Modules
-------
attention  plain softmax attention (forward and backward) written from its
           definition; full, row-sampled and key-sampled variants.
schedule   the 2D mesh coordinates, paired-block (zigzag) placement and the
           inner/outer double-ring step table.
ring       a second, chunked oracle that walks the ring schedule block pair by
           block pair and merges the partial results by log-sum-exp.
merge      n-way log-sum-exp merge of partial attention outputs.
repack     the Ulysses head-context layout repack (S/P,H) <-> (S,H/P).

Sources (page title, section):
  [G]  "Guide to LoongTrain: 2D Head-Context Parallelism for LLMs"
  [A]  "LoongTrain: Efficient Training of Long-Sequence LLMs with
       Head-Context Parallelism" (paper abstract page)
Where the pages leave a step open the plain reading is taken; each such
reading is named in the docstring of the function that relies on it.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms, finite differences, library special cases
or the pages' printed formulas.
"""
