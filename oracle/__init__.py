"""CPU oracle for the sharded ZeRO optimizer step.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the package smoke check and
by bench.py's CPU-baseline leg.  The product (the CUDA library and its Python
binding) never imports it.
"""
