"""GB300 (sm_103a) implementation of the Kimi Delta Attention (KDA) layer."""
