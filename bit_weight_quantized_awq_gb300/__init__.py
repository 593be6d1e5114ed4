"""GB300 (sm_103a) AWQ W4A16 linear forward (placeholder while the binding is written)."""
