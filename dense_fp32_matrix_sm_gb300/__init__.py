"""GB300-native FP32 SGEMM: C = alpha*A*B + beta*C on row-major float32 matrices."""
