// nvfp4_internal.cuh -- the NVFP4 quantiser's block pass as a library-internal
// host call (defined in nvfp4.cu), for callers that have the tensor amax
// already (the NVFP4 FFN takes it in GEMM1's epilogue).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_r3.h"

namespace moe {

// src [rows, cols] bf16 (cols % 16 == 0, 16-byte aligned); tensor_scale[1]
// holds the tensor amax on entry, tensor_scale[0] receives s_enc; q [rows,
// cols/2] and scales [rows, cols/16] as fp8_quant_nvfp4 writes them.
moe_status nvfp4_quant_blocks(const uint16_t *src, int64_t rows, int64_t cols, float *tensor_scale, uint8_t *q,
                              uint8_t *scales, cudaStream_t stream);

} // namespace moe
