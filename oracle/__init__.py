"""Test infrastructure: the plain CPU oracle of the folded verification layer.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg import this package; the product path never does.
"""
