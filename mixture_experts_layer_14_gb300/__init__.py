"""GB300-native (sm_103a) DeepSeek-V3-style MoE layer: Python binding of the C-ABI library."""
