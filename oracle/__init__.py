"""CPU oracle of the DFlash drafter forward: test infrastructure only (see dflash_oracle)."""
