"""CPU oracle of the staged halo exchange (test infrastructure only)."""
