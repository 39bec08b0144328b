"""Row-wise normalization reduce for GB300 (sm_103a)."""
