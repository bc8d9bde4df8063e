"""fp64 CPU oracle for decode attention (test infrastructure only).

This package is the checker, not the product. Only the test suite, the
smoke check in ``__graft_entry__`` and the ``cpu_baseline`` / reference
arm of ``bench.py`` may import it. The CUDA path never imports it and it
never imports the CUDA path: the two share no code, tables or helpers.

Contents
--------
``cost``       analytic FLOP / byte / arithmetic-intensity counter and the
               KV-cache size accounting of the pages.
``attention``  plain NumPy float64 definitions of grouped-head decode
               attention (MHA / GQA / MQA), absorbed latent MLA (absorb,
               latent attention, output projection), the expanded MLA
               brute force, the log-sum-exp merge of split partials and the
               paged-cache gather.

Every input is widened exactly from bf16 to float64 by the caller; no
intermediate is rounded. Each function names the passage it follows.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against something other than itself (a library routine, a closed form,
an algebraic identity, brute force on tiny inputs, or numbers the pages
print). None is "parity unpinned".
"""
