// launch.h -- host-side entry points of the kernels, called by fa_api.cu after
// argument validation.  Each returns an FA_* code.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

// Row softmax of x [rows, N] into y (y may equal x).
int launch_softmax_rows(const float *x, float *y, int64_t rows, int64_t N, cudaStream_t stream);

// Arguments shared by both attention paths.  Layout rules are those of fa.h.
struct AttnArgs {
    const void *Q, *K, *V;
    void *O;
    float *lse;
    int B, H, N, d;
    int64_t total;            // packed token count (B * N when dense)
    float scale;
    int causal;
    const int32_t *cu_seqlens;  // device pointer or nullptr (dense)
    int *err_word;            // device error word
};

int launch_attention_bf16(const AttnArgs &a, cudaStream_t stream);
int launch_attention_f32(const AttnArgs &a, cudaStream_t stream);

}  // namespace fa
