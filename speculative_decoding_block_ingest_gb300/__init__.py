"""GB300-native DFlash block-diffusion drafter round (ingest + gamma=16 block forward)."""
