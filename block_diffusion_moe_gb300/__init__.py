"""GB300-native hot path of block-diffusion decoding in a Clover-shaped MoE."""
