"""mmact: fused GEMM / implicit-GEMM conv with a bias + activation epilogue on GB300."""
