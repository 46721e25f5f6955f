// Device twin of the seeded input generator in synth/__init__.py.  It holds
// none of the method's arithmetic: it only fills tensors with the same bits
// the host generator produces (SplitMix64 mixer, Irwin-Hall(12) of 16-bit
// fields, one fp32 multiply, round to nearest even into the storage type).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <typename T> __device__ __forceinline__ T cvt(float v);
template <> __device__ __forceinline__ float cvt<float>(float v) { return v; }
template <> __device__ __forceinline__ __half cvt<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T>
__global__ void fill_kernel(T *dst, long long rows, long long cols, long long ld, uint64_t key, float scale) {
    const long long total = rows * ld;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / ld, col = i - row * ld;
        float v = 0.f;
        if (col < cols) {
            const uint64_t n = (uint64_t)(row * cols + col);
            int s = 0;
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const uint64_t r = mix64(key + (3ull * n + (uint64_t)k + 1ull) * kGamma);
                s += (int)(r & 0xFFFF) + (int)((r >> 16) & 0xFFFF) + (int)((r >> 32) & 0xFFFF) +
                     (int)((r >> 48) & 0xFFFF);
            }
            v = __fmul_rn((float)(s - 393210), scale);
        }
        dst[i] = cvt<T>(v);
    }
}

}  // namespace

extern "C" {

// Stream key of a tensor: mix64(seed * G + mix64(tensor_id)).
unsigned long long synth_stream_key(unsigned long long seed, unsigned long long tid) {
    return mix64(seed * kGamma + mix64(tid));
}

// Fill dst [rows, ld] (dtype 0 f32, 1 f16, 2 bf16) with the N(0, std^2) tensor
// (seed, tid); columns >= cols are zero.  scale = float32(std * 2^-16).
int synth_fill_normal(void *dst, int dtype, long long rows, long long cols, long long ld,
                      unsigned long long seed, unsigned long long tid, float scale, void *stream) {
    if (!dst || rows < 0 || cols < 0 || ld < cols) return 1;
    if (rows == 0 || ld == 0) return 0;
    const uint64_t key = synth_stream_key(seed, tid);
    const long long total = rows * ld;
    long long blocks = (total + 255) / 256;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    cudaStream_t s = (cudaStream_t)stream;
    switch (dtype) {
    case 0: fill_kernel<float><<<(unsigned)blocks, 256, 0, s>>>((float *)dst, rows, cols, ld, key, scale); break;
    case 1: fill_kernel<__half><<<(unsigned)blocks, 256, 0, s>>>((__half *)dst, rows, cols, ld, key, scale); break;
    case 2: fill_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>((__nv_bfloat16 *)dst, rows, cols, ld, key, scale); break;
    default: return 1;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"
