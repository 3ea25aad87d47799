"""Plain CPU oracle of the CacheGen KV-cache codec (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline and
reference arm may import this package.  It shares no code with the product.
"""
