"""fp64 CPU oracle for masked attention over a BlockMask. TEST INFRASTRUCTURE ONLY: imported by tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg, never by the library."""
