// CUDA twin of synth.py's mixture generator: the same SplitMix64 counters,
// the same Irwin-Hall normals and the same fp64 operations in the same order
// (explicit _rn intrinsics: no contraction into FMA), so it writes the same
// bf16 bytes as the numpy side.  Input generation only; no codec arithmetic.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr double kNormScale = 0x1.bb67ae8584caap-16;   // sqrt(3) / 65536

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * kGamma); }

__device__ __forceinline__ double normal(uint64_t h) {
    int64_t s = (int64_t)(h & 0xFFFF) + (int64_t)((h >> 16) & 0xFFFF) + (int64_t)((h >> 32) & 0xFFFF) +
                (int64_t)(h >> 48);
    return __dmul_rn((double)(s - 131070), kNormScale);
}

struct UnitKeys {
    uint64_t centers, assign, drift, noise;
    uint64_t outlier_mask[4];
};

// tab[h][f][m][d]: centres per frame, drifting frame by frame.
__global__ void center_table_kernel(const UnitKeys* keys, int M, int D, int F, double drift_std, double* tab) {
    const int h = blockIdx.y;
    const int64_t md = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (md >= (int64_t)M * D) return;
    const UnitKeys k = keys[h];
    double* t = tab + (int64_t)h * F * M * D;
    double v = normal(draw(k.centers, (uint64_t)md));
    t[md] = v;
    for (int f = 1; f < F; ++f) {
        const double z = normal(draw(k.drift, (uint64_t)f * M * D + md));
        v = __dadd_rn(v, __dmul_rn(drift_std, z));
        t[(int64_t)f * M * D + md] = v;
    }
}

__global__ void mixture_kernel(const UnitKeys* keys, const double* tab, int M, int D, int F, int frame_tokens,
                               int64_t tok_begin, int64_t n_tokens, double noise_std, double factor,
                               uint16_t* out, int64_t head_stride, int64_t token_stride) {
    const int h = blockIdx.y;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_tokens * D) return;
    const int64_t r = i / D;
    const int d = (int)(i % D);
    const int64_t n = tok_begin + r;
    const UnitKeys k = keys[h];
    const int m = (int)(draw(k.assign, (uint64_t)n) % (uint64_t)M);
    const int f = (int)(n / frame_tokens);
    const double z = normal(draw(k.noise, (uint64_t)n * D + d));
    double x = __dadd_rn(tab[(((int64_t)h * F + f) * M + m) * D + d], __dmul_rn(noise_std, z));
    if ((k.outlier_mask[d >> 6] >> (d & 63)) & 1ull) x = __dmul_rn(x, factor);
    const float xf = __double2float_rn(x);
    out[(int64_t)h * head_stride + r * token_stride + d] = __bfloat16_as_ushort(__float2bfloat16_rn(xf));
}

}  // namespace

extern "C" {

// keys: device array of H UnitKeys; tab: device scratch of H*F*M*D doubles.
__attribute__((visibility("default"))) int synth_mixture(const void* keys, int H, int M, int D, int F,
                                                         int frame_tokens, int64_t tok_begin, int64_t n_tokens,
                                                         double noise_std, double drift_std, double factor,
                                                         double* tab, uint16_t* out, int64_t head_stride,
                                                         int64_t token_stride, void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    const UnitKeys* k = (const UnitKeys*)keys;
    const int64_t md = (int64_t)M * D;
    center_table_kernel<<<dim3((unsigned)((md + 255) / 256), (unsigned)H), 256, 0, s>>>(k, M, D, F, drift_std, tab);
    const int64_t total = n_tokens * D;
    if (total > 0)
        mixture_kernel<<<dim3((unsigned)((total + 255) / 256), (unsigned)H), 256, 0, s>>>(
            k, tab, M, D, F, frame_tokens, tok_begin, n_tokens, noise_std, factor, out, head_stride, token_stride);
    return (int)cudaGetLastError();
}

}  // extern "C"
