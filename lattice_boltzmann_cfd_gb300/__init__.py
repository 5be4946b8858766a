"""GB300-native lattice-Boltzmann collide-and-stream step (placeholder; filled below)."""
