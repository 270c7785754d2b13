"""Float64 CPU oracle of the GRPO loss path (test infrastructure only)."""
