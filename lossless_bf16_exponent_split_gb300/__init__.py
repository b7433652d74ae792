"""lossless_bf16_exponent_split_gb300 -- GB300 lossless BF16 exponent codec."""
