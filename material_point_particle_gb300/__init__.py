"""GB300-native MPM particle/grid transfer (placeholder until the binding lands)."""
