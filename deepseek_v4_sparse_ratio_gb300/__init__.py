"""DeepSeek-V4 indexed sparse attention for chunked prefill, on one GB300 (sm_103a)."""
