/*
 * Device twin of gen.c: the same counter-based SplitMix64 hash and Box-Muller transform in
 * double precision, evaluated on the GPU so that multi-gigabyte synthetic weights and KV
 * caches can be drawn straight into device memory. Element i of a (seed, stream) pair is
 * the same function of i as in gen.c; only the double-precision log / sin / cos / sqrt
 * come from the device's math library instead of the host's, so a value can differ from
 * the host's only where those differ by an ulp right at a bf16 rounding boundary.
 *
 * Like gen.c, this file holds nothing of the offloading method: it produces input data.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

__host__ __device__ static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN_GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL + 1ULL));
}

__device__ static inline uint16_t to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

__global__ void normal_bf16_kernel(uint64_t key, double mean, double std, uint64_t offset, uint64_t n,
                                   uint16_t* out) {
    for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n; j += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t i = offset + j;
        const uint64_t r = mix64(key + ((i >> 1) + 1ULL) * GOLDEN_GAMMA);
        const double u1 = ((double)(r >> 32) + 0.5) * (1.0 / 4294967296.0);
        const double u2 = ((double)(r & 0xFFFFFFFFULL) + 0.5) * (1.0 / 4294967296.0);
        const double rad = sqrt(-2.0 * log(u1));
        const double ang = 6.283185307179586476925286766559 * u2;
        const double z = (i & 1ULL) ? rad * sin(ang) : rad * cos(ang);
        out[j] = to_bf16((float)(mean + std * z));
    }
}

/* out (device) [j] = bf16(mean + std * N(0,1)_{offset + j}), j < n; asynchronous on stream.
 * Returns 0 or the CUDA error code. */
extern "C" int synth_dev_normal_bf16(uint64_t seed, uint64_t stream, double mean, double std, uint64_t offset,
                                     uint64_t n, void* out, void* cuda_stream) {
    if (n == 0) return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint64_t blocks = (n + 255) / 256;
    const uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 16;
    if (blocks > cap) blocks = cap;
    normal_bf16_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(stream_key(seed, stream), mean, std,
                                                                                  offset, n, (uint16_t*)out);
    return (int)cudaGetLastError();
}
