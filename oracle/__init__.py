"""fp64 CPU oracle of the draft-verification sampler -- TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's cpu-baseline / reference
leg may import this package.  The product package never does.
"""
