"""Plain CPU oracle for the MPM transfer path (test infrastructure only).

Loaded by the test suite, ``__graft_entry__`` and the benchmark's CPU-baseline
leg; the CUDA library never imports, links or calls anything here.
"""
