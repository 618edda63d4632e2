"""f64 CPU oracle of the KDA / Gated DeltaNet mixer.  Test infrastructure only: imported by the
test suite, the smoke check and the benchmark's CPU-baseline leg, never by the product path."""
