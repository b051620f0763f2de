"""GB300-native DCP LSE-weighted merge for MLA decode (placeholder until the binding lands)."""
