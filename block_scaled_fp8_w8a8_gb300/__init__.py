"""GB300-native (sm_103a) W8A8 block-FP8 matmul."""
