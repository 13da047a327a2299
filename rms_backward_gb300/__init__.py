"""GB300-native mHC projection/RMS backward (sm_103a CUDA kernels behind a C-ABI)."""
