"""fp64 CPU oracle of the TSP layer. Test infrastructure only: imported by tests/,
the package smoke check and the benchmark's CPU-baseline leg, never by the library."""
