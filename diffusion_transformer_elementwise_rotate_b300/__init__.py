"""B300-native elementwise hot path of a diffusion-transformer block."""
