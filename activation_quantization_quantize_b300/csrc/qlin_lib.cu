// qlin_lib.cu -- single translation unit of libqlin.so (the kernels share
// device-side state such as the error word, so they are compiled together).
#include "quantize.cu"
#include "gemm_w8a8.cu"
#include "gemm_w4a16.cu"
#include "gemm_w4a8.cu"
#include "calib.cu"
#include "llmint8.cu"
#include "kvcache.cu"
#include "api.cu"
#include "noalloc.cu"
