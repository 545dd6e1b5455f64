"""GB300 dense GEMM library (C-ABI) and its Python binding."""
