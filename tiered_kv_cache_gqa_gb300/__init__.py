"""tkv: tiered KV-cache decode attention for one GB300 (sm_103a)."""
