// synth_fill.cu -- device side of the seeded input generator (synth.py).
//
// Not part of the verify walk: it only draws synthetic inputs on the GPU so that
// large workloads need no host generation.  Every value equals, bit for bit, the
// one synth.py draws for the same key and element index on the CPU:
//   out(c)  = SplitMix64 finaliser of key + (c + 1) * golden-ratio increment
//             (Steele, Lea and Flood, 2014, as published with SplitMix64)
//   normal  = (sum of the twelve 16-bit fields of out(3n), out(3n+1), out(3n+2)
//              - 393210) * 2^-16, then one f32 multiply by sigma
//   uniform = ((out(n) >> 40) - 2^23) * 2^-24, then one f32 multiply by 2*half_width
//   bf16    = round-to-nearest-even of the f32 value's top 16 bits
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t out_c(uint64_t key, uint64_t c) { return mix(key + (c + 1) * GAMMA); }

__device__ __forceinline__ void store(void *out, int bf16, size_t e, float x)
{
    if (bf16) {
        uint32_t u = __float_as_uint(x);
        u = u + 0x7FFFu + ((u >> 16) & 1u);
        static_cast<uint16_t *>(out)[e] = static_cast<uint16_t>(u >> 16);
    } else {
        static_cast<float *>(out)[e] = x;
    }
}

__global__ void normal_kernel(uint64_t key, uint64_t start, size_t n, float sigma, int scale, int bf16, void *out)
{
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const uint64_t idx = start + e;
        int64_t total = 0;
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const uint64_t r = out_c(key, 3 * idx + m);
#pragma unroll
            for (int f = 0; f < 4; ++f)
                total += static_cast<int64_t>((r >> (16 * f)) & 0xFFFFull);
        }
        float z = __fmul_rn(static_cast<float>(total - 393210), 1.52587890625e-05f);  // 2^-16
        if (scale)
            z = __fmul_rn(z, sigma);
        store(out, bf16, e, z);
    }
}

__global__ void uniform_kernel(uint64_t key, uint64_t start, size_t n, float factor, int scale, int bf16, void *out)
{
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const int64_t u = static_cast<int64_t>(out_c(key, start + e) >> 40);
        float x = __fmul_rn(static_cast<float>(u - (1ll << 23)), 5.9604644775390625e-08f);  // 2^-24
        if (scale)
            x = __fmul_rn(x, factor);
        store(out, bf16, e, x);
    }
}

unsigned grid_for(size_t n)
{
    size_t g = (n + 255) / 256;
    return static_cast<unsigned>(g > 152 * 64 ? 152 * 64 : (g < 1 ? 1 : g));
}

}  // namespace

extern "C" int synth_fill_normal(uint64_t key, uint64_t start, size_t n, float sigma, int bf16, void *out,
                                 cudaStream_t stream)
{
    if (n == 0)
        return 0;
    normal_kernel<<<grid_for(n), 256, 0, stream>>>(key, start, n, sigma, sigma != 1.0f, bf16, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int synth_fill_uniform(uint64_t key, uint64_t start, size_t n, float half_width, int bf16, void *out,
                                  cudaStream_t stream)
{
    if (n == 0)
        return 0;
    const float factor = 2.0f * half_width;
    uniform_kernel<<<grid_for(n), 256, 0, stream>>>(key, start, n, factor, half_width != 0.5f, bf16, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
