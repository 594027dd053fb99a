"""CPU oracle (test infrastructure only; never imported by the product path).

``oracle.oracle`` is the fp64 NumPy oracle, ``oracle.brute`` an independent
pure-Python brute force used to pin it on tiny cases.
"""
