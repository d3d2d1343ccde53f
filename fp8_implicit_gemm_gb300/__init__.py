"""FP8 (e4m3) implicit-GEMM 3D convolution with a BF16 NCDHW output, for one GB300 (sm_103a)."""
