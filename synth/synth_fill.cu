// synth_fill.cu -- device-side filler for the seeded synthetic inputs.
//
// Same SplitMix64 counter generator as synth/__init__.py (Steele, Lea & Flood,
// OOPSLA 2014), used only to fill large expert sets quickly on the GPU.  It is
// input generation, not part of the method: no kernel of the MoE library and
// no part of the oracle includes or calls it.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// byte i of the stream lives in output word (offset + i) / 8, byte (offset + i) % 8
__global__ void fill_bytes_kernel(uint8_t* dst, uint64_t n, uint64_t key, uint64_t offset)
{
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        uint64_t b = offset + i;
        uint64_t w = mix64(key + (b / 8 + 1) * kGamma);
        dst[i] = (uint8_t)(w >> (8 * (b % 8)));
    }
}

// fast path: 8-byte aligned destination and offset, whole words
__global__ void fill_words_kernel(uint64_t* dst, uint64_t nwords, uint64_t key, uint64_t word0)
{
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nwords; i += stride)
        dst[i] = mix64(key + (word0 + i + 1) * kGamma);
}

__global__ void fill_range_kernel(uint8_t* dst, uint64_t n, uint64_t key, uint64_t offset,
                                  uint32_t lo, uint32_t span)
{
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        uint64_t r = mix64(key + (offset + i + 1) * kGamma) >> 32;
        dst[i] = (uint8_t)(lo + ((r * span) >> 32));
    }
}

uint64_t stream_key(uint64_t seed, uint64_t stream) { return mix64(seed * kGamma + stream); }

int grid_for(uint64_t n)
{
    uint64_t g = (n + 255) / 256;
    return (int)(g > 8192 ? 8192 : (g ? g : 1));
}

}  // namespace

extern "C" int synth_fill_bytes(void* dst, uint64_t n, uint64_t seed, uint64_t stream,
                                uint64_t offset, void* cuda_stream)
{
    if (!dst && n) return -1;
    if (!n) return 0;
    cudaStream_t s = (cudaStream_t)cuda_stream;
    uint64_t key = stream_key(seed, stream);
    if (((uintptr_t)dst % 8 == 0) && (offset % 8 == 0) && (n % 8 == 0)) {
        uint64_t nw = n / 8;
        fill_words_kernel<<<grid_for(nw), 256, 0, s>>>((uint64_t*)dst, nw, key, offset / 8);
    } else {
        fill_bytes_kernel<<<grid_for(n), 256, 0, s>>>((uint8_t*)dst, n, key, offset);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

extern "C" int synth_fill_range(void* dst, uint64_t n, uint64_t seed, uint64_t stream,
                                uint64_t offset, int lo, int hi, void* cuda_stream)
{
    if ((!dst && n) || hi < lo || lo < 0 || hi > 255) return -1;
    if (!n) return 0;
    uint64_t key = stream_key(seed, stream);
    fill_range_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
        (uint8_t*)dst, n, key, offset, (uint32_t)lo, (uint32_t)(hi - lo + 1));
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
