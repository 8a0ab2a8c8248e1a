"""GB300-native F^H D / Q gather for iterative non-Cartesian MRI reconstruction."""
