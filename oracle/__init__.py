"""fp64 CPU oracle for hybrid local/global GQA attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the benchmark's CPU-baseline / reference leg.  The product library
never imports it and shares no code with it.
"""
