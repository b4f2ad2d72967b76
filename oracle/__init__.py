"""CPU oracle for paged KV-cache decode — test infrastructure only.

Imported only by the tests, by the package smoke check and by the benchmark's
CPU-baseline leg. The product path never imports it.
"""
