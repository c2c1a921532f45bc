"""GB300 (sm_103a) NVFP4 mixture-of-experts FFN forward behind a C-ABI library."""
