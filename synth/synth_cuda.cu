// synth_cuda.cu — device half of the seeded input generator (definition in
// include/mk_synth.h).  Written independently of synth.c from the same
// published splitmix64 definition; tests compare the two bit for bit.
#include <cstdint>
#include <cuda_runtime.h>

#include "mk_synth.h"

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}

__device__ __forceinline__ uint16_t normal_value(uint64_t u, float c, float offset) {
    int32_t s = static_cast<int32_t>(u & 0xFFFF) + static_cast<int32_t>((u >> 16) & 0xFFFF) +
                static_cast<int32_t>((u >> 32) & 0xFFFF) + static_cast<int32_t>(u >> 48);
    float z = __fmul_rn(static_cast<float>(s - 131070), c);  // no fusion with the add
    return to_bf16_rne(__fadd_rn(offset, z));
}

__global__ void fill_normal_kernel(uint16_t* out, int64_t n, uint64_t key, uint64_t i0, float c, float offset) {
    int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < n; j += stride) {
        uint64_t u = mix64(key + (i0 + static_cast<uint64_t>(j) + 1) * kGolden);
        out[j] = normal_value(u, c, offset);
    }
}

__global__ void fill_kv_pages_kernel(uint16_t* pool, const int32_t* page_table, int32_t batch, int32_t max_pages,
                                     int32_t ctx, int32_t nkv, int32_t page_size, int32_t hd, uint64_t key, float c) {
    int64_t n = static_cast<int64_t>(batch) * ctx * nkv * hd;
    int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        int32_t e = static_cast<int32_t>(i % hd);
        int32_t h = static_cast<int32_t>((i / hd) % nkv);
        int64_t bt = i / (static_cast<int64_t>(hd) * nkv);
        int32_t t = static_cast<int32_t>(bt % ctx);
        int32_t b = static_cast<int32_t>(bt / ctx);
        int32_t page = page_table[static_cast<int64_t>(b) * max_pages + t / page_size];
        int64_t dst = ((static_cast<int64_t>(page) * nkv + h) * page_size + (t % page_size)) * hd + e;
        uint64_t u = mix64(key + (static_cast<uint64_t>(i) + 1) * kGolden);
        pool[dst] = normal_value(u, c, 0.0f);
    }
}

uint64_t host_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

int grid_for(int64_t n) {
    int64_t g = (n + 255) / 256;
    return static_cast<int>(g > 148 * 32 ? 148 * 32 : (g < 1 ? 1 : g));
}

}  // namespace

extern "C" int mk_synth_normal_bf16_device(uint16_t* out, int64_t n, uint64_t seed, uint64_t tid, uint64_t i0,
                                           float c, float offset, void* stream) {
    if (!out || n < 0) return -1;
    if (n == 0) return 0;
    uint64_t key = host_mix64(seed + (tid + 1) * kGolden);
    fill_normal_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(out, n, key, i0, c, offset);
    return static_cast<int>(cudaGetLastError());
}

extern "C" int mk_synth_kv_pages_device(uint16_t* pool, const int32_t* page_table, int32_t batch, int32_t max_pages,
                                        int32_t ctx, int32_t n_kv_heads, int32_t page_size, int32_t head_dim,
                                        uint64_t seed, uint64_t tid, float c, void* stream) {
    if (!pool || !page_table || batch <= 0 || max_pages <= 0 || ctx < 0 || n_kv_heads <= 0 || page_size <= 0 ||
        head_dim <= 0 || ctx > max_pages * page_size)
        return -1;
    if (ctx == 0) return 0;
    uint64_t key = host_mix64(seed + (tid + 1) * kGolden);
    int64_t n = static_cast<int64_t>(batch) * ctx * n_kv_heads * head_dim;
    fill_kv_pages_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        pool, page_table, batch, max_pages, ctx, n_kv_heads, page_size, head_dim, key, c);
    return static_cast<int>(cudaGetLastError());
}
