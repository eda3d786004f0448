"""fp64 CPU oracle for the fused SDPA forward -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline
leg may import this package.  See ``oracle.oracle`` and ``sdpa_oracle.c``.
"""
