"""Row-wise top-k (RTop-K) and the MaxK layer on GB300 (sm_103a)."""
