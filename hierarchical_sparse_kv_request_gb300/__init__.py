"""HiSparse decode-time swap-in resolver for GB300 (sm_103a)."""
