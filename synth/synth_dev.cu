// Counter-based synthetic input generator, GPU side. Same definition as
// synth_host.c (see there); used to fill large weight tensors in device memory
// without a host round trip. Holds none of the MoE layer's arithmetic.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27; z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

__device__ __forceinline__ float draw(uint64_t key, uint64_t i, int dist, float K) {
    uint64_t r = mix64(key + (i + 1) * 0x9E3779B97F4A7C15ULL);
    int32_t n;
    if (dist == 0) {
        uint32_t s = (uint32_t)(r & 0xFFFF) + (uint32_t)((r >> 16) & 0xFFFF) +
                     (uint32_t)((r >> 32) & 0xFFFF) + (uint32_t)(r >> 48);
        n = 2 * (int32_t)s - 262140;
    } else {
        n = 2 * (int32_t)(r >> 41) - ((1 << 23) - 1);
    }
    return __fmul_rn((float)n, K);
}

__global__ void fill_kernel(uint64_t key, uint64_t offset, uint64_t count, int dist, float K,
                            int out_bf16, void* out) {
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride) {
        float v = draw(key, offset + j, dist, K);
        if (out_bf16) ((__nv_bfloat16*)out)[j] = __float2bfloat16_rn(v);
        else ((float*)out)[j] = v;
    }
}

uint64_t host_mix64(uint64_t z) {
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27; z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

}  // namespace

extern "C" int synth_dev_fill(uint64_t seed, uint64_t tid, uint64_t offset, uint64_t count,
                              int dist, float K, int out_bf16, void* out, cudaStream_t stream) {
    if (count == 0) return 0;
    uint64_t key = host_mix64((seed + 1) * 0x9E3779B97F4A7C15ULL + tid * 0xD1B54A32D192ED03ULL);
    uint64_t blocks = (count + 255) / 256;
    if (blocks > 148ull * 64) blocks = 148ull * 64;
    fill_kernel<<<(unsigned)blocks, 256, 0, stream>>>(key, offset, count, dist, K, out_bf16, out);
    return (int)cudaGetLastError();
}
