"""Importance-weighted GGML IQ codebook encoder, decoder and per-expert imatrix for B300."""
