"""GB300-native two-stage quantized MoE expert computation (sort, stage 1, stage 2)."""
