"""Float64 oracle of the TTT-E2E inner loop: test infrastructure, never a product path."""
