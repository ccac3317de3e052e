"""GB300-native dense GEMM: D = act(alpha * (A @ B) + beta * C) on sm_103a."""
