"""CPU oracle for the VQ3 MLP path. Test infrastructure only: imported by tests/,
__graft_entry__.smoke() and the benchmark's CPU-baseline leg, never by the library."""
