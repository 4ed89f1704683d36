"""CPU oracle of the P-EAGLE drafting step: test infrastructure only.

Imported by the tests, the smoke check and the benchmark's CPU-baseline leg;
never by the library or its Python binding.
"""
