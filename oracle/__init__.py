"""fp64 CPU oracle of the decode MoE expert block: test infrastructure, not product code."""
