"""Plain fp64 CPU oracle for the ReplaySSM decode path.

TEST INFRASTRUCTURE ONLY.  This package is the independent checker that the
CUDA path is compared against.  Only the test suite, the package smoke check
(``__graft_entry__.smoke``) and the CPU-baseline leg of ``bench.py`` may import
it.  The product path (the C-ABI library and its Python binding) never imports,
links or calls anything here, and nothing here imports the product path: the
two share only the seeded input generators, which hold no arithmetic of the
method.

Source of truth: the web page "ReplaySSM: Cache SSM Inputs, Not State"
(papercache summary of Tri Dao's blog post); for the convolution state that
precedes the SSM (``conv.py``), the state layout of "Disaggregated Serving for
Hybrid SSM Models".  Each function names the section and equation it follows.  Everything is computed in float64 with numpy, as
plainly as the equations are written; loops over sequences and buffer entries
are explicit.

Pins (what ties this code to something other than itself) live in
``tests/test_oracle_*.py``: agreement between the page's independent forms
(summary route vs history route vs output-only route; Householder form vs
rank-1 form; chunked triangular solve vs serial recurrence), flush-schedule
and rollback invariants, closed forms, exact scalar examples and brute force.
"""
