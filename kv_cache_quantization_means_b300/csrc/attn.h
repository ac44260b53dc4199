// Attention over a compressed K/V history (see attn.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qvg {

struct AttnArgs {
    const uint16_t* q;                  // bf16, q + h*q_head_stride + i*q_token_stride
    int64_t q_head_stride, q_token_stride, n_queries;
    const uint32_t *k_codes, *k_meta;   // [S][H][cap][D*bits/32], [S][H][cap][D/G]
    const uint32_t *v_codes, *v_meta;
    const uint8_t *k_ids, *v_ids;       // [H][cap] (C > 0)
    const uint16_t *k_cent, *v_cent;    // bf16 [H][C][D] (C > 0)
    int64_t cap, n_keys;
    float* out;                         // fp32, out + h*out_head_stride + i*out_token_stride
    int64_t out_head_stride, out_token_stride;
    int H, C, S, G, bits;
    float scale_log2;                   // softmax scale * log2(e), rounded to fp32
};

// Launches the fused decode + attention kernel (D = 64 or 128).  Returns
// cudaErrorInvalidValue for any other head dimension or code width.
cudaError_t launch_attention_decode(int D, const AttnArgs& a, cudaStream_t s);

// The tensor-core path (attn_tc.cu): groups of kAttnGroupHeads heads decoded
// into a working buffer of attention_staged_bytes, then attended.  D = 128;
// *launched = false (cudaSuccess) when the shape, layout or buffer is outside
// what it handles.
constexpr int kAttnGroupHeads = 4;
size_t attention_staged_bytes(int D, int H, int64_t n_keys);
cudaError_t launch_attention_staged(int D, const AttnArgs& a, void* ws, size_t ws_bytes, bool* launched,
                                    cudaStream_t s);

}  // namespace qvg
