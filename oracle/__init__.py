"""CPU oracle of the MoE layer (float64 numpy). Test infrastructure only: the
library never imports it; the tests, the smoke check and the benchmark's CPU
baseline do."""
