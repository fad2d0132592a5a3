"""libfattn: exact IO-aware attention on GB300 (sm_103a)."""
